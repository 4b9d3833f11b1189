"""Pins of the per-tensor FP8 oracle (dynamic scaling, one scale per tensor).

None of these re-evaluates the quantizer's own expression: nearest-code brute
force, the exact landing of the largest element on 448, the special case that
coincides with the MX quantizer, power-of-two equivariance, the error bound,
and the grouped forward against independent one-expert runs.
"""
import numpy as np
import pytest

from oracle import expert_ffn as ef
from oracle import fp8_tensor as pt
from oracle import mxfp8 as mx
from oracle import routing as rt


def _bf16_tensor(rng, shape, std):
    return mx.bf16(rng.standard_normal(shape) * std)


ALL_VALUES = mx.e4m3_decode(np.arange(256))


def _nearest_code_brute_force(y):
    """Nearest finite E4M3 value to y (ties to the even code), saturating at +-448."""
    finite = ~np.isnan(ALL_VALUES)
    codes = np.arange(256)[finite]
    vals = ALL_VALUES[finite]
    out = np.zeros(y.shape, dtype=np.int64)
    for i, v in np.ndenumerate(y):
        d = np.abs(vals - v)
        best = codes[d == d.min()]
        if len(best) > 1:                            # ties go to the even code ...
            best = [c for c in best if c % 2 == 0]
            if all(ALL_VALUES[c] == 0 for c in best):  # ... and a zero keeps the sign of v
                best = [0x80 if np.signbit(v) else 0x00]
        out[i] = best[0]
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_codes_are_the_nearest_values_of_the_scaled_tensor(seed):
    rng = np.random.default_rng(seed)
    v = _bf16_tensor(rng, (6, 40), 10.0 ** rng.uniform(-3, 3))
    codes, s = pt.quantize_tensor(v)
    y = (v.astype(np.float32) * np.float32(s)).astype(np.float64)
    assert np.array_equal(codes.astype(np.int64), _nearest_code_brute_force(y))


@pytest.mark.parametrize("seed", range(6))
def test_the_largest_magnitude_lands_on_448(seed):
    rng = np.random.default_rng(10 + seed)
    v = _bf16_tensor(rng, (33, 17), 10.0 ** rng.uniform(-6, 6))
    codes, s = pt.quantize_tensor(v)
    dec = mx.e4m3_decode(codes)
    assert np.max(np.abs(dec)) == 448.0
    i = np.unravel_index(np.argmax(np.abs(v)), v.shape)
    assert abs(dec[i]) == 448.0


def test_zero_tensor_has_unit_scale_and_zero_codes():
    codes, s = pt.quantize_tensor(np.zeros((4, 8)))
    assert s == 1.0 and not codes.any()


@pytest.mark.parametrize("j", [-20, -3, 0, 5])
def test_power_of_two_scale_coincides_with_the_mx_quantizer(j):
    """amax = 448 * 2^j: s = 2^-j, the MX block scale of a block holding that amax."""
    rng = np.random.default_rng(j + 50)
    v = _bf16_tensor(rng, (4, 32), 2.0 ** j * 100)
    v[2, 7] = np.ldexp(448.0, j)
    codes, s = pt.quantize_tensor(v)
    assert s == np.ldexp(1.0, -j)
    mc, ms = mx.quantize_blocks(v, axis=-1)
    assert np.array_equal(ms[2], [j + 127])
    assert np.array_equal(codes[2], mc[2])


@pytest.mark.parametrize("m", [-7, 3])
def test_power_of_two_equivariance(m):
    rng = np.random.default_rng(77)
    v = _bf16_tensor(rng, (8, 64), 1.0)
    c0, s0 = pt.quantize_tensor(v)
    c1, s1 = pt.quantize_tensor(np.ldexp(v, m))
    assert np.array_equal(c0, c1) and s1 == np.ldexp(s0, -m)


@pytest.mark.parametrize("seed", [3, 4])
def test_error_within_half_an_e4m3_step(seed):
    rng = np.random.default_rng(seed)
    v = _bf16_tensor(rng, (16, 64), 0.5)
    deq, s = pt.qdq(v)
    # normal E4M3 range: half a step is 2^-4 relative; subnormals: 2^-10 absolute (scaled units);
    # the float32 product adds at most 2^-24 relative before the rounding
    bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 / s) * (1 + 2.0 ** -20)
    assert np.all(np.abs(deq - v) <= bound)


def _workload(seed, T=48, H=64, I=96, E=4, k=2):
    rng = np.random.default_rng(seed)
    x = _bf16_tensor(rng, (T, H), 1.0)
    w_gu = _bf16_tensor(rng, (E, 2 * I, H), 0.05)
    w_d = _bf16_tensor(rng, (E, H, I), 0.05)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 0] += 2.0 * rng.standard_normal(T).astype(np.float32)   # uneven loads
    idx, prob = rt.route_topk(logits, k)
    return x, idx, prob.astype(np.float64), w_gu, w_d


def test_grouped_forward_equals_independent_one_expert_runs():
    """Every expert's scales come from its own operands only."""
    x, idx, prob, w_gu, w_d = _workload(0)
    E = w_gu.shape[0]
    full = pt.forward(x, idx, prob, w_gu, w_d)
    perm = full["perm"]
    for e in range(E):
        r0, m = int(perm["offsets_pad"][e]), int(perm["split_sizes"][e])
        if m == 0:
            continue
        toks = perm["src_of"][r0:r0 + m]
        slot_p = full["prob_perm"][r0:r0 + m]
        one = pt.forward(x[toks], np.zeros((m, 1), dtype=np.int32), slot_p[:, None], w_gu[e:e + 1], w_d[e:e + 1])
        assert np.array_equal(one["y"][:m], full["y"][r0:r0 + m])
        assert one["s_x"][0] == full["s_x"][e] and one["s_a"][0] == full["s_a"][e]


def test_power_of_two_down_weights_scale_the_output_exactly():
    x, idx, prob, w_gu, w_d = _workload(1)
    base = pt.forward(x, idx, prob, w_gu, w_d)["out"]
    scaled = pt.forward(x, idx, prob, w_gu, np.ldexp(w_d, 5))["out"]
    assert np.array_equal(scaled, np.ldexp(base, 5))


def test_close_to_the_unquantized_forward_and_different_from_it():
    x, idx, prob, w_gu, w_d = _workload(2)
    q = pt.forward(x, idx, prob, w_gu, w_d)["out"]
    ref = ef.forward(x, idx, prob, w_gu, w_d, ef.UNQUANTIZED_BF16)["out"]
    rel = np.linalg.norm(q - ref) / np.linalg.norm(ref)
    assert 1e-3 < rel < 0.1


def test_expert_scales_differ_so_one_global_scale_would_fail_the_pins():
    """The workload's experts see different amax, so a single shared scale is caught above."""
    x, idx, prob, w_gu, w_d = _workload(0)
    full = pt.forward(x, idx, prob, w_gu, w_d)
    used = full["perm"]["split_sizes"] > 0
    assert len(set(full["s_x"][used])) > 1 and len(set(full["s_a"][used])) > 1
    assert len(set(full["wq"]["gu_s"])) > 1


def _workload_bwd(seed):
    x, idx, prob, w_gu, w_d = _workload(seed)
    dout = _bf16_tensor(np.random.default_rng(seed + 100), x.shape, 0.01)
    return x, idx, prob, w_gu, w_d, dout


def test_backward_close_to_the_exact_backward_and_different_from_it():
    x, idx, prob, w_gu, w_d, dout = _workload_bwd(5)
    got = pt.backward(pt.forward(x, idx, prob, w_gu, w_d), dout)
    ex = ef.backward(ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT), dout, ef.EXACT)
    for key in ("dx", "dw_gu", "dw_d", "dprob"):
        rel = np.linalg.norm(got[key] - ex[key]) / np.linalg.norm(ex[key])
        assert 1e-3 < rel < 0.15, (key, rel)


def test_power_of_two_dout_scales_every_gradient_exactly():
    """dY, dA, dH are linear in dout and every per-tensor scale follows its tensor, so a 2^m
    factor on dout passes through every quantizer unchanged."""
    x, idx, prob, w_gu, w_d, dout = _workload_bwd(6)
    fwd = pt.forward(x, idx, prob, w_gu, w_d)
    base = pt.backward(fwd, dout)
    scaled = pt.backward(fwd, np.ldexp(dout, 4))
    for key in ("dx", "dw_gu", "dw_d"):
        assert np.array_equal(scaled[key], np.ldexp(base[key], 4)), key
    assert np.allclose(scaled["dprob"], np.ldexp(base["dprob"], 4), rtol=1e-6)


def test_backward_of_grouped_equals_independent_one_expert_runs():
    x, idx, prob, w_gu, w_d, dout = _workload_bwd(7)
    full_f = pt.forward(x, idx, prob, w_gu, w_d)
    full = pt.backward(full_f, dout)
    perm = full_f["perm"]
    for e in range(w_gu.shape[0]):
        r0, m = int(perm["offsets_pad"][e]), int(perm["split_sizes"][e])
        if m == 0:
            continue
        toks = perm["src_of"][r0:r0 + m]
        p = full_f["prob_perm"][r0:r0 + m][:, None]
        one_f = pt.forward(x[toks], np.zeros((m, 1), dtype=np.int32), p, w_gu[e:e + 1], w_d[e:e + 1])
        one = pt.backward(one_f, dout[toks])
        assert np.array_equal(one["dw_gu"][0], full["dw_gu"][e])
        assert np.array_equal(one["dw_d"][0], full["dw_d"][e])

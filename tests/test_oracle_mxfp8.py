"""Pins of the oracle's MXFP8 codec against brute force, closed forms and hand examples."""
import os

import numpy as np
import pytest

from oracle import mxfp8 as mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return bits.view(np.float32).astype(np.float64)


def e4m3_table():
    """All 127 non-negative finite E4M3 values (codes 0x00..0x7E), from decode."""
    codes = np.arange(0x7F, dtype=np.uint8)
    return codes, mx.e4m3_decode(codes)


def brute_force_encode(y):
    """Nearest finite E4M3 value by exhaustive search; ties -> even code."""
    y = np.asarray(y, dtype=np.float64)
    codes, vals = e4m3_table()
    a = np.abs(y)
    out = np.empty(y.shape, dtype=np.int64)
    flat_a, flat_o = a.ravel(), out.ravel()
    for s in range(0, flat_a.size, 8192):
        blk = flat_a[s:s + 8192]
        d = np.abs(blk[:, None] - vals[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        # prefer even codes among ties: score = tie * (2 if even else 1)
        score = cand * (1 + (codes[None, :] % 2 == 0))
        flat_o[s:s + 8192] = np.argmax(score, axis=1)
    return (out | (np.signbit(y).astype(np.int64) << 7)).astype(np.uint8)


def check_encode_exhaustive(encode=mx.e4m3_encode):
    """Every bf16 pattern times a sweep of power-of-two factors: encode == brute force."""
    v = all_bf16_values()
    v = v[np.isfinite(v)]
    bad = 0
    for sh in range(-140, 140, 7):
        y = np.ldexp(v, sh)
        y = y[np.abs(y) < 1e6]
        bad += int(np.count_nonzero(encode(y) != brute_force_encode(y)))
    return bad


def test_decode_definition_points():
    assert mx.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert mx.e4m3_decode(np.uint8(0x38)) == 1.0
    assert mx.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6
    assert mx.e4m3_decode(np.uint8(0x07)) == 7 * 2.0 ** -9
    assert np.isnan(mx.e4m3_decode(np.uint8(0x7F))) and np.isnan(mx.e4m3_decode(np.uint8(0xFF)))
    z = mx.e4m3_decode(np.uint8(0x80))
    assert z == 0.0 and np.signbit(z)
    # monotone over the positive codes, and sign symmetric
    _, vals = e4m3_table()
    assert np.all(np.diff(vals) > 0)
    codes = np.arange(0x7F, dtype=np.uint8)
    assert np.array_equal(mx.e4m3_decode(codes | 0x80), -vals)


def test_encode_equals_brute_force_all_bf16():
    assert check_encode_exhaustive() == 0


def test_encode_golden_hand_examples():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_hand_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((float(parts[0]), int(parts[1], 16)))
    vals = np.array([r[0] for r in rows])
    want = np.array([r[1] for r in rows], dtype=np.uint8)
    got = mx.e4m3_encode(vals)
    assert np.array_equal(got, want), list(zip(vals, got, want))


def test_half_step_bound_and_idempotence():
    v = all_bf16_values()
    v = v[np.isfinite(v)]
    for sh in (-120, -12, -8, 0, 5):
        y = np.ldexp(v, sh)
        y = y[np.abs(y) <= 448.0]
        q = mx.e4m3_encode(y)
        d = mx.e4m3_decode(q)
        # spacing of the E4M3 grid at |y|
        _, ex = np.frexp(np.where(y == 0, 1.0, np.abs(y)))
        step = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
        assert np.all(np.abs(d - y) <= 0.5 * step)
        assert np.array_equal(mx.e4m3_encode(d), q)                 # idempotent
        assert np.array_equal(mx.e4m3_encode(-y), q ^ np.uint8(0x80))  # sign symmetric


def test_scale_rule_closed_form_and_minimality():
    rng = np.random.default_rng(1)
    amax = np.abs(rng.standard_normal(20000)) * np.exp2(rng.integers(-140, 120, 20000))
    amax = amax.astype(np.float32).astype(np.float64)
    e = mx.scale_exponent(amax)
    assert np.all(amax <= np.ldexp(448.0, e))                 # never saturates
    unclamped = e > -127
    r = amax[unclamped] / np.ldexp(1.0, e[unclamped])
    assert np.all((r > 224.0) & (r <= 448.0))                 # closed form interval
    # brute force over every representable exponent on a subset
    for a, ee in zip(amax[:300], e[:300]):
        ok = [x for x in range(-127, 128) if a <= 448.0 * 2.0 ** x]
        assert ee == ok[0]


def test_scale_golden_hand_examples():
    with open(os.path.join(GOLDEN, "mx_scale_hand_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a_txt, code, *_ = line.split()
            a = float.fromhex(a_txt) if a_txt.startswith("0x") else float(a_txt)
            a = float(np.float32(a))
            assert int(mx.scale_exponent(a)) + 127 == int(code), a_txt


def test_block_example_and_one_scale_per_32():
    blk = np.zeros(32)
    blk[:3] = [1.0, -0.5, np.float32(0.1)]
    codes, sc = mx.quantize_blocks(blk[None, :], axis=-1)
    assert sc.shape == (1, 1) and sc[0, 0] == 119
    assert list(codes[0, :4]) == [0x78, 0xF0, 0x5D, 0x00]
    # shape: one scale per 32 consecutive values along the chosen axis
    x = np.random.default_rng(2).standard_normal((64, 96)).astype(np.float32).astype(np.float64)
    c0, s0 = mx.quantize_blocks(x, axis=1)
    c1, s1 = mx.quantize_blocks(x, axis=0)
    assert s0.shape == (64, 3) and s1.shape == (2, 96)
    # changing one element only touches its own block
    x2 = x.copy()
    x2[5, 40] *= 1000.0
    c2, s2 = mx.quantize_blocks(x2, axis=1)
    diff_blocks = np.argwhere(s2 != s0)
    assert diff_blocks.tolist() == [[5, 1]]
    changed = np.argwhere(c2 != c0)
    assert np.all(changed[:, 0] == 5) and np.all((changed[:, 1] >= 32) & (changed[:, 1] < 64))


def test_zero_and_nonfinite_blocks():
    x = np.zeros((2, 64))
    x[1, 33] = np.inf
    c, s = mx.quantize_blocks(x, axis=1)
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0 and s[1, 1] == 255
    assert np.all(c[0] == 0) and np.all(c[1, :32] == 0) and np.all(c[1, 32:] == 0x7F)


def test_dequantize_within_step_of_input():
    """dequantize(quantize(x)) stays within half an E4M3 step of x (scaled back)."""
    x = np.random.default_rng(3).standard_normal((128, 256)) * 3.0
    x = x.astype(np.float32).astype(np.float64)
    c, s = mx.quantize_blocks(x, axis=1)
    d = mx.dequantize_blocks(c, s, axis=1)
    e = np.repeat(s.astype(np.int64) - 127, 32, axis=1)
    y = np.ldexp(np.abs(x), -e)
    _, ex = np.frexp(np.where(y == 0, 1.0, y))
    step = np.ldexp(np.ldexp(1.0, np.maximum(ex - 1, -6) - 3), e)
    assert np.all(np.abs(d - x) <= 0.5 * step)


def test_bf16_rounding_helper():
    # bf16 keeps 7 explicit mantissa bits: the spacing at 1.0 is 2^-7
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 0.0])
    got = mx.bf16(f)
    assert list(got) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.5, 0.0]


@pytest.mark.parametrize("mutation", ["half_up", "truncate"])
def test_planted_rounding_mistakes_are_caught(monkeypatch, mutation):
    """A plausible rounding mistake in the encoder fails the exhaustive pin."""
    real_round = np.round

    def half_up(v):
        return np.floor(v + 0.5)

    def truncate(v):
        return np.trunc(v)

    bad_round = {"half_up": half_up, "truncate": truncate}[mutation]

    def mutated(y):
        monkeypatch.setattr(np, "round", bad_round)
        try:
            return mx.e4m3_encode(y)
        finally:
            monkeypatch.setattr(np, "round", real_round)

    assert check_encode_exhaustive(mutated) > 0


def test_planted_scale_mistake_is_caught(monkeypatch):
    """Taking e = floor(log2 amax) - 8 without the saturation check breaks the closed form."""
    def floor_only(amax):
        amax = np.asarray(amax, dtype=np.float64)
        _, ex = np.frexp(np.where(amax == 0, 1.0, amax))
        return np.clip(ex - 1 - 8, -127, 127)
    amax = np.array([1.8, 449.0, 3.9], dtype=np.float64)
    assert not np.all(amax <= np.ldexp(448.0, floor_only(amax)))
    assert np.all(amax <= np.ldexp(448.0, mx.scale_exponent(amax)))

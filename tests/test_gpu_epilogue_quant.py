"""The GEMM epilogues' MX quantizer, bit for bit against the oracle's codec.

The epilogues quantize float32 values with full 24-bit significands (a after
ScaledSwiGLU, dH after the SwiGLU backward; page "Efficient MoE Training for
Biological Foundation Models", section "MXFP8与融合MLP").  Inside the layer
their inputs differ from the oracle's by accumulation order, so the layer
tests compare those codes only after dequantization.  Here the very device
functions the epilogues call (through moe_selftest_epilogue_quant) get the
oracle's OWN float32 a and dH, and values placed on the scale rule's
1.75 * 2^E boundary and on E4M3 rounding ties; every code and scale must
equal the oracle's, along rows and along tokens.
"""
import numpy as np
import pytest
import torch

from helpers import untile_scales
from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build, configs, synth
from oracle import expert_ffn as ef
from oracle import mxfp8 as mx
from oracle import routing as rt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def run_device(v32):
    """Row-wise and along-token (transposed) MX codes of a float32 [rows][cols] array."""
    rows, cols = v32.shape
    src = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).cuda()
    codes = torch.full((rows, cols), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows * cols // 32,), 0xA5, dtype=torch.uint8, device="cuda")
    codes_t = torch.full((cols, rows), 0xA5, dtype=torch.uint8, device="cuda")
    scales_t = torch.full((rows * cols // 32,), 0xA5, dtype=torch.uint8, device="cuda")
    B.moe_selftest_epilogue_quant(src, rows, cols, codes, scales, codes_t, scales_t)
    torch.cuda.synchronize()
    return (codes.cpu().numpy(), untile_scales(scales.cpu().numpy(), rows, cols),
            codes_t.cpu().numpy(), untile_scales(scales_t.cpu().numpy(), cols, rows))


def check_bit_exact(v32, name):
    v = np.asarray(v32, dtype=np.float32).astype(np.float64)
    c, s, ct, st = run_device(v32)
    ref_c, ref_s = mx.quantize_blocks(v, axis=1)
    assert np.array_equal(s, ref_s), f"{name}: row scales"
    assert np.array_equal(c, ref_c), f"{name}: row codes ({np.count_nonzero(c != ref_c)} differ)"
    ref_c, ref_s = mx.quantize_blocks(v, axis=0)
    assert np.array_equal(st, ref_s.T), f"{name}: token scales"
    assert np.array_equal(ct, ref_c.T), f"{name}: token codes ({np.count_nonzero(ct != ref_c.T)} differ)"


def oracle_intermediates(wl):
    inp = synth.make_inputs(wl, 0)
    f64 = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    idx, prob = rt.route_topk(inp["logits"].numpy(), wl.k)
    fwd = ef.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]), ef.MXFP8)
    bwd = ef.backward(fwd, f64(inp["dout"]), ef.MXFP8)
    return fwd["a"], bwd["dH"]


@pytest.mark.parametrize("wl", [configs.get(configs.TINY),
                                configs.small(300, 256, 384, 6, 2, routing="biased", backward=True)],
                         ids=["tiny", "ragged_T300_I384_E6"])
def test_oracle_a_and_dH_quantize_identically(wl):
    a, dH = oracle_intermediates(wl)
    # the oracle's quantizer inputs are float32 values (rounded from its float64 arithmetic)
    assert np.array_equal(mx.fp32(a), a) and np.array_equal(mx.fp32(dH), dH)
    check_bit_exact(a.astype(np.float32), "a")
    check_bit_exact(dH.astype(np.float32), "dH")


def f32_from_bits(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def test_scale_boundary_and_rounding_ties():
    """Hand-placed float32 values (128 x 128): block maxima with significand 1.75 (0x600000,
    the largest that keeps e = E - 8) and one ulp above it; elements that sit exactly half
    way between two E4M3 codes after scaling (ties to even), in the normal and the
    subnormal range; one ulp either side of a tie; signed zeros; all-zero blocks; and
    random full-significand values with random exponents."""
    rng = np.random.default_rng(11)
    v = np.zeros((128, 128), dtype=np.float32)
    exps = rng.integers(-20, 20, size=(128, 4))
    for r in range(128):
        for b in range(4):
            blk = slice(32 * b, 32 * b + 32)
            kind = (r + b) % 6
            E = int(exps[r, b])
            if kind == 0:                                   # max exactly 1.75 * 2^E
                top = f32_from_bits([((E + 127) << 23) | 0x600000])[0]
            elif kind == 1:                                 # one ulp above 1.75 * 2^E
                top = f32_from_bits([((E + 127) << 23) | 0x600001])[0]
            elif kind == 2:                                 # exactly 448 * 2^(E-8) scale: max = 2^E
                top = np.float32(2.0 ** E)
            else:
                top = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** E)
            row = rng.standard_normal(32).astype(np.float32) * np.float32(top) / np.float32(4.0)
            row[0] = top if r % 2 == 0 else -top
            # with top in (224, 448] * 2^e, the scale is 2^e, e = E - 8 (+1 above 1.75)
            e = E - 8 + (1 if kind == 1 else 0)
            sc = np.float32(2.0 ** e)
            # ties between E4M3 codes in the normal range: (1 + (2m + 1)/16) * 2^j
            for t, (m, j) in enumerate([(0, 0), (1, 0), (2, 3), (3, -4), (5, 5), (6, -6)]):
                row[1 + t] = np.float32((1.0 + (2 * m + 1) / 16.0) * 2.0 ** j) * sc
            # ties in the subnormal range (step 2^-9): (2m + 1) * 2^-10
            for t, m in enumerate([0, 1, 2, 3, 6]):
                row[7 + t] = np.float32((2 * m + 1) * 2.0 ** -10) * sc * (1 if t % 2 else -1)
            # one float32 ulp either side of a tie
            tie = np.float32(1.0625 * 2.0 ** 2) * sc
            row[12] = np.nextafter(tie, np.float32(np.inf))
            row[13] = np.nextafter(tie, np.float32(-np.inf))
            row[14] = np.float32(-0.0)
            row[15] = np.float32(0.0)
            # a value that rounds up into the next binade: 1.9375 + 1 ulp of E4M3's half step
            row[16] = np.float32(1.96875 * 2.0 ** 1) * sc
            if kind == 5 and r % 3 == 0:
                row[:] = 0.0                                # all-zero block
                row[5] = np.float32(-0.0)
            v[r, blk] = row
    # the right half: random float32 with random exponents and full significands
    bits = (rng.integers(0, 1 << 23, size=(128, 64), dtype=np.int64)
            | ((rng.integers(90, 170, size=(128, 64), dtype=np.int64)) << 23)
            | (rng.integers(0, 2, size=(128, 64), dtype=np.int64) << 31)).astype(np.uint32)
    v[:, 64:] = bits.view(np.float32)
    assert np.all(np.isfinite(v))
    check_bit_exact(v, "hand-placed")
    check_bit_exact(np.ascontiguousarray(v.T), "hand-placed, transposed")


def test_host_checks():
    z = torch.zeros(128, 96, dtype=torch.float32, device="cuda")
    u8 = torch.zeros(128 * 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoeError):
        B.moe_selftest_epilogue_quant(z, 128, 96, u8, u8, u8, u8)

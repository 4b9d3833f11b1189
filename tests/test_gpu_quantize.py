"""GPU mxfp8_quantize vs the oracle codec: bit-exact codes and scales."""
import numpy as np
import pytest
import torch

from helpers import untile_scales
from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build
from oracle import mxfp8 as mx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def bf16_from_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16)


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_quant(x: torch.Tensor, batch: int, rows: int, cols: int, axis: int):
    xd = x.cuda().contiguous()
    codes = torch.empty(x.numel(), dtype=torch.uint8, device="cuda")
    scales = torch.full((x.numel() // 32,), 0xAB, dtype=torch.uint8, device="cuda")
    B.mxfp8_quantize(xd, batch, rows, cols, axis, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def all_patterns_matrix(seed: int) -> np.ndarray:
    """Every bf16 bit pattern once (sorted or shuffled), as a [512][128] matrix."""
    bits = np.arange(65536, dtype=np.uint32)
    if seed:
        bits = np.random.default_rng(seed).permutation(bits)
    return bits.reshape(512, 128)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_rowwise_every_bf16_pattern(seed):
    bits = all_patterns_matrix(seed)
    x = bf16_from_bits(bits)
    codes, scales = run_quant(x, 1, 512, 128, 0)
    with np.errstate(invalid="ignore"):
        ref_c, ref_s = mx.quantize_blocks(as_f64(x), axis=1)
    got_s = untile_scales(scales, 512, 128)
    assert np.array_equal(got_s, ref_s), np.argwhere(got_s != ref_s)[:5]
    bad = np.argwhere(codes.reshape(512, 128) != ref_c)
    assert bad.size == 0, [(tuple(i), hex(bits[tuple(i)]), codes.reshape(512, 128)[tuple(i)], ref_c[tuple(i)])
                           for i in bad[:8]]


@pytest.mark.parametrize("seed", [0, 5])
def test_colwise_every_bf16_pattern(seed):
    bits = all_patterns_matrix(seed)
    x = bf16_from_bits(bits)
    codes, scales = run_quant(x, 1, 512, 128, 1)
    with np.errstate(invalid="ignore"):
        ref_c, ref_s = mx.quantize_blocks(as_f64(x), axis=0)     # blocks along rows
    got_c = codes.reshape(128, 512)                               # transposed
    got_s = untile_scales(scales, 128, 512)
    assert np.array_equal(got_s, ref_s.T)
    assert np.array_equal(got_c, ref_c.T)


def test_colwise_many_tiles():
    """A 16384 x 1024 matrix along its rows: 2048 gathered tiles of 128 x 64, each filling
    one half of its scale atoms.  Random bf16 bit patterns (NaN, Inf, zeros and
    subnormals among them) and whole NaN and subnormal blocks, compared with the oracle."""
    rows, cols = 16384, 1024
    bits = np.random.default_rng(11).integers(0, 65536, size=(rows, cols), dtype=np.uint32)
    bits[:32, :5] = 0x7FC0                                        # whole NaN blocks
    bits[32:64, 7] = 0x0001                                       # a block of the smallest subnormal
    x = bf16_from_bits(bits)
    codes, scales = run_quant(x, 1, rows, cols, 1)
    with np.errstate(invalid="ignore"):
        ref_c, ref_s = mx.quantize_blocks(as_f64(x), axis=0)
    assert np.array_equal(untile_scales(scales, cols, rows), ref_s.T)
    assert np.array_equal(codes.reshape(cols, rows), ref_c.T)


@pytest.mark.parametrize("scale_pow", [-60, -20, 0, 12])
def test_batched_weights_both_axes(scale_pow):
    E, R, C = 3, 256, 384
    g = torch.Generator().manual_seed(scale_pow + 100)
    w = (torch.randn(E, R, C, generator=g) * (2.0 ** scale_pow)).to(torch.bfloat16)
    w[1, 5, :64] = 0                                              # all-zero blocks
    w[2, :32, 7] = 0
    wf = as_f64(w)
    codes, scales = run_quant(w, E, R, C, 0)
    ref_c, ref_s = mx.quantize_blocks(wf, axis=2)
    assert np.array_equal(codes.reshape(E, R, C), ref_c)
    assert np.array_equal(untile_scales(scales, E * R, C), ref_s.reshape(E * R, C // 32))
    codes, scales = run_quant(w, E, R, C, 1)
    ref_c, ref_s = mx.quantize_blocks(wf, axis=1)
    assert np.array_equal(codes.reshape(E, C, R), np.swapaxes(ref_c, 1, 2))
    assert np.array_equal(untile_scales(scales, E * C, R), np.swapaxes(ref_s, 1, 2).reshape(E * C, R // 32))


def test_dual_equals_the_two_single_axis_calls():
    E, R, C = 3, 256, 384
    g = torch.Generator().manual_seed(7)
    w = (torch.randn(E, R, C, generator=g) * 0.02).to(torch.bfloat16).cuda()
    w[0, 3, :] = 0
    c0 = torch.empty(E * R * C, dtype=torch.uint8, device="cuda")
    s0 = torch.empty(E * R * C // 32, dtype=torch.uint8, device="cuda")
    c1, s1 = torch.empty_like(c0), torch.empty_like(s0)
    d0, t0, d1, t1 = (torch.empty_like(c0), torch.empty_like(s0), torch.empty_like(c0), torch.empty_like(s0))
    B.mxfp8_quantize(w, E, R, C, 0, c0, s0)
    B.mxfp8_quantize(w, E, R, C, 1, c1, s1)
    B.mxfp8_quantize_dual(w, E, R, C, d0, t0, d1, t1)
    torch.cuda.synchronize()
    assert torch.equal(c0, d0) and torch.equal(s0, t0) and torch.equal(c1, d1) and torch.equal(s1, t1)


@pytest.mark.parametrize("seed", [0, 9])
def test_dual_every_bf16_pattern(seed):
    """Both orientations of one read, on every bf16 bit pattern (NaN, Inf, zeros, subnormals)."""
    bits = all_patterns_matrix(seed)
    x = bf16_from_bits(bits).cuda()
    codes = torch.empty(65536, dtype=torch.uint8, device="cuda")
    scales = torch.empty(2048, dtype=torch.uint8, device="cuda")
    codes_t, scales_t = torch.empty_like(codes), torch.empty_like(scales)
    B.mxfp8_quantize_dual(x, 1, 512, 128, codes, scales, codes_t, scales_t)
    torch.cuda.synchronize()
    with np.errstate(invalid="ignore"):
        rc, rs = mx.quantize_blocks(as_f64(x), axis=1)
        cc, cs = mx.quantize_blocks(as_f64(x), axis=0)
    assert np.array_equal(codes.cpu().numpy().reshape(512, 128), rc)
    assert np.array_equal(untile_scales(scales.cpu().numpy(), 512, 128), rs)
    assert np.array_equal(codes_t.cpu().numpy().reshape(128, 512), cc.T)
    assert np.array_equal(untile_scales(scales_t.cpu().numpy(), 128, 512), cs.T)


@pytest.mark.parametrize("both", [True, False])
def test_per_expert_pointers_equal_the_stacked_tensor(both):
    """One tensor per expert, allocated separately, gives the stacked results bit for bit."""
    E, R, C = 5, 256, 384
    g = torch.Generator().manual_seed(11)
    experts = [(torch.randn(R, C, generator=g) * 0.02 * (e + 1)).to(torch.bfloat16).cuda() for e in range(E)]
    pad = [torch.empty(1000 + 37 * e, dtype=torch.uint8, device="cuda") for e in range(E)]   # scatter the allocations
    stacked = torch.stack(experts)
    c0 = torch.empty(E * R * C, dtype=torch.uint8, device="cuda")
    s0 = torch.empty(E * R * C // 32, dtype=torch.uint8, device="cuda")
    c1, s1 = torch.empty_like(c0), torch.empty_like(s0)
    d0, t0, d1, t1 = (torch.full_like(c0, 0xEE), torch.full_like(s0, 0xEE), torch.full_like(c0, 0xEE),
                      torch.full_like(s0, 0xEE))
    B.mxfp8_quantize_dual(stacked, E, R, C, c0, s0, c1, s1)
    if both:
        B.mxfp8_quantize_experts(experts, R, C, d0, t0, d1, t1)
    else:
        B.mxfp8_quantize_experts(experts, R, C, d0, t0)
    torch.cuda.synchronize()
    assert torch.equal(c0, d0) and torch.equal(s0, t0)
    if both:
        assert torch.equal(c1, d1) and torch.equal(s1, t1)
    else:
        assert bool((d1 == 0xEE).all()) and bool((t1 == 0xEE).all())   # untouched
    del pad


def test_per_tensor_per_expert_pointers_equal_the_stacked_tensor():
    E, R, C = 4, 128, 256
    g = torch.Generator().manual_seed(12)
    experts = [(torch.randn(R, C, generator=g) * 10.0 ** (e - 2)).to(torch.bfloat16).cuda() for e in range(E)]
    stacked = torch.stack(experts)
    c0 = torch.empty(E, R, C, dtype=torch.uint8, device="cuda")
    c1 = torch.empty_like(c0)
    a0 = torch.empty(E, dtype=torch.float32, device="cuda")
    a1 = torch.empty_like(a0)
    B.fp8_tensor_quantize(stacked, E, R, C, c0, a0)
    B.fp8_tensor_quantize_experts(experts, R, C, c1, a1)
    torch.cuda.synchronize()
    assert torch.equal(c0, c1) and torch.equal(a0, a1)

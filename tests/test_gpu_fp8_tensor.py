"""Per-tensor FP8 forward (one dynamic scale per expert operand tensor) vs its oracle.

Bit-exact: the E4M3 codes and amax of the weights and of x's permuted rows
(identical inputs on both sides).  Within the float tolerance: the bf16
activation a, its codes after dequantization, amax of a, y and out -- their
inputs differ by the GEMMs' accumulation order.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close
from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN
from oracle import fp8_tensor as pt
from oracle import mxfp8 as mx
from oracle import routing as rt

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("error::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_weight_codes_and_amax_bit_exact():
    g = torch.Generator().manual_seed(3)
    E, R, C = 3, 256, 384
    w = (torch.randn(E, R, C, generator=g) * torch.tensor([0.02, 3.0, 1e-4]).view(E, 1, 1)).to(torch.bfloat16)
    w[1, 7, 9] = -50.0                                   # one dominant element
    w[2, :, :128] = 0
    wd = w.cuda()
    codes = torch.empty(E, R, C, dtype=torch.uint8, device="cuda")
    amax = torch.empty(E, dtype=torch.float32, device="cuda")
    B.fp8_tensor_quantize(wd, E, R, C, codes, amax)
    torch.cuda.synchronize()
    for e in range(E):
        ref_c, ref_s = pt.quantize_tensor(f64(w[e]))
        assert np.array_equal(codes[e].cpu().numpy(), ref_c)
        assert float(amax[e]) == float(np.max(np.abs(f64(w[e]))))
        assert pt.tensor_scale(float(amax[e])) == ref_s


def test_all_zero_tensor_has_unit_scale():
    w = torch.zeros(2, 128, 128, dtype=torch.bfloat16, device="cuda")
    w[1, 3, 4] = 1.0
    codes = torch.full((2, 128, 128), 0x55, dtype=torch.uint8, device="cuda")
    amax = torch.full((2,), 7.0, dtype=torch.float32, device="cuda")
    B.fp8_tensor_quantize(w, 2, 128, 128, codes, amax)
    torch.cuda.synchronize()
    assert amax.tolist() == [0.0, 1.0]
    assert not codes[0].any()
    assert int(codes[1, 3, 4]) == 0x7E and int(codes[1].count_nonzero()) == 1     # 448 = S.1111.110


@pytest.mark.parametrize("name_or_dims", [
    configs.TINY,
    (300, 256, 384, 6, 2, "biased"),
    (513, 384, 640, 5, 3, "normal"),
    (700, 256, 256, 16, 4, "biased"),
    (600, 128, 128, 256, 8, "biased"),
    configs.UNEVEN,
])
def test_fp8_tensor_forward_matches_oracle(name_or_dims):
    wl = configs.get(name_or_dims) if isinstance(name_or_dims, str) else configs.small(*name_or_dims[:5],
                                                                                         routing=name_or_dims[5])
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0, with_grad=False).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=False)
    L.route(inp["logits"], inp["x"])
    L.quantize_weights_fp8_tensor(inp["w_gu"], inp["w_d"])
    out = L.forward_fp8_tensor(inp["x"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)

    idx, prob = rt.route_topk(inp["logits"].cpu().numpy(), wl.k)
    w_gu, w_d = f64(inp["w_gu"]), f64(inp["w_d"])
    fwd = pt.forward(f64(inp["x"]), idx, prob.astype(np.float64), w_gu, w_d)
    perm, rows = fwd["perm"], fwd["perm"]["rows"]
    used = perm["split_sizes"] > 0

    # weights and x: bit-exact codes and scales
    wq = fwd["wq"]
    assert np.array_equal(L.t8_wgu.cpu().numpy(), wq["gu"])
    assert np.array_equal(L.t8_wd.cpu().numpy(), wq["d"])
    assert [pt.tensor_scale(v) for v in L.t8_amax_gu.cpu().tolist()] == list(wq["gu_s"])
    assert [pt.tensor_scale(v) for v in L.t8_amax_d.cpu().tolist()] == list(wq["d_s"])
    s_x = np.array([pt.tensor_scale(v) for v in L.t8_amax_x.cpu().tolist()])
    assert np.array_equal(s_x[used], fwd["s_x"][used])
    assert np.array_equal(L.t8_xq.cpu().numpy()[:rows], fwd["xq_codes"])

    # the activation and what follows: float tolerance
    assert_close(f64(L.t8_a[:rows]), fwd["a"], "a (bf16)")
    s_a = np.array([pt.tensor_scale(v) for v in L.t8_amax_a.cpu().tolist()])
    assert np.allclose(s_a[used], fwd["s_a"][used], rtol=2e-2)
    offs = perm["offsets_pad"]
    aq_dev = np.zeros((rows, wl.I))
    aq_ref = np.zeros((rows, wl.I))
    codes = L.t8_aq.cpu().numpy()
    for e in np.nonzero(used)[0]:
        sl = slice(int(offs[e]), int(offs[e]) + int(perm["split_sizes"][e]))
        aq_dev[sl] = pt.dequantize_tensor(codes[sl], s_a[e])
        aq_ref[sl] = pt.dequantize_tensor(fwd["aq_codes"][sl], fwd["s_a"][e])
    assert_close(aq_dev, aq_ref, "a after per-tensor quantization")
    assert_close(f64(L.t8_y[:rows]), fwd["y"], "y")
    assert_close(f64(out), fwd["out"], "out")


def test_padding_rows_of_x_are_zero_codes():
    """Padding rows are rewritten to zero codes on every call (stale NaN codes planted first)."""
    wl = configs.small(300, 256, 256, 6, 2, routing="biased", backward=False)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0, with_grad=False).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=False)
    L.route(inp["logits"], inp["x"])
    L.quantize_weights_fp8_tensor(inp["w_gu"], inp["w_d"])
    L.forward_fp8_tensor(inp["x"])
    L.t8_xq.fill_(0x7F)
    out = L.forward_fp8_tensor(inp["x"])
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    split = L.split_sizes.cpu().numpy()
    xq = L.t8_xq.cpu().numpy()
    r0 = 0
    for m in split:
        pad = (-int(m)) % 128
        assert not xq[r0 + m:r0 + m + pad].any()
        r0 += int(m) + pad
    assert not np.isnan(mx.e4m3_decode(xq[:r0])).any()


@pytest.mark.parametrize("name_or_dims", [
    configs.TINY,
    (300, 256, 384, 6, 2, "biased"),
    (513, 384, 640, 5, 3, "normal"),
    (600, 128, 128, 256, 8, "biased"),
])
def test_fp8_tensor_training_step_matches_oracle(name_or_dims):
    """Per-tensor FP8 forward (saving g, u) + backward vs the oracle's per-tensor backward."""
    wl = configs.get(name_or_dims) if isinstance(name_or_dims, str) else configs.small(*name_or_dims[:5],
                                                                                         routing=name_or_dims[5])
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0, with_grad=True).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=True)
    L.route(inp["logits"], inp["x"])
    L.quantize_weights_fp8_tensor(inp["w_gu"], inp["w_d"])
    L.forward_fp8_tensor(inp["x"])
    dx = L.backward_fp8_tensor(inp["dout"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    idx, prob = rt.route_topk(inp["logits"].cpu().numpy(), wl.k)
    fwd = pt.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]))
    bwd = pt.backward(fwd, f64(inp["dout"]))
    rows, I = fwd["perm"]["rows"], wl.I
    assert_close(f64(L.saved_gu[:rows, :I]), fwd["g"], "g")
    assert_close(f64(L.saved_gu[:rows, I:]), fwd["u"], "u")
    assert_close(f64(dx), bwd["dx"], "dx")
    assert_close(f64(L.t8_dwgu), bwd["dw_gu"], "dW_gu")
    assert_close(f64(L.t8_dwd), bwd["dw_d"], "dW_d")
    assert_close(L.t8_dprob.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob")


def test_per_tensor_codes_do_not_depend_on_the_axis():
    """Codes of the transposed tensor are the transposed codes: the byte transposes of the
    per-tensor backward give the along-token operands exactly."""
    g = torch.Generator().manual_seed(8)
    w = (torch.randn(2, 256, 384, generator=g) * 0.1).to(torch.bfloat16).cuda()
    codes = torch.empty(2, 256, 384, dtype=torch.uint8, device="cuda")
    amax = torch.empty(2, dtype=torch.float32, device="cuda")
    B.fp8_tensor_quantize(w, 2, 256, 384, codes, amax)
    wt = w.transpose(1, 2).contiguous()
    codes_t = torch.empty(2, 384, 256, dtype=torch.uint8, device="cuda")
    amax_t = torch.empty(2, dtype=torch.float32, device="cuda")
    B.fp8_tensor_quantize(wt, 2, 384, 256, codes_t, amax_t)
    torch.cuda.synchronize()
    assert torch.equal(amax, amax_t) and torch.equal(codes.transpose(1, 2), codes_t)

"""GPU expert-FFN layer vs the oracle on the same seeded inputs.

Bit-exact: routing indices, split_sizes, the permutation, the MX codes and
scales of x (both axes).  Floats (y, saved g/u, a after quantization along
tokens, out, dx, dW_gu, dW_d, dprob): relative Frobenius error <= 5e-3 and
max abs error <= 2e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close, rel_frob, untile_scales
from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN
from oracle import expert_ffn as ef
from oracle import mxfp8 as mx
from oracle import routing as rt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(wl, inp, training):
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=training)
    dev = {k: v.cuda() for k, v in inp.items()}
    L.quantize_weights(dev["w_gu"], dev["w_d"])
    L.forward(dev["logits"], dev["x"])
    if training:
        L.backward(dev["dout"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    return L


def run_oracle(wl, inp, training):
    idx, prob = rt.route_topk(inp["logits"].numpy(), wl.k)
    x, w_gu, w_d = f64(inp["x"]), f64(inp["w_gu"]), f64(inp["w_d"])
    fwd = ef.forward(x, idx, prob.astype(np.float64), w_gu, w_d, ef.MXFP8)
    bwd = ef.backward(fwd, f64(inp["dout"]), ef.MXFP8) if training else None
    return idx, prob, fwd, bwd


def check_layer(wl, inp, training, report=None):
    L = run_gpu(wl, inp, training)
    idx, prob, fwd, bwd = run_oracle(wl, inp, training)
    perm = fwd["perm"]
    rows = perm["rows"]
    # ---- bit-exact routing and permutation ----
    assert np.array_equal(L.idx.cpu().numpy(), idx)
    assert np.allclose(L.prob.cpu().numpy(), prob, rtol=2e-6, atol=1e-7)
    assert np.array_equal(L.split_sizes.cpu().numpy(), perm["split_sizes"])
    assert np.array_equal(L.row_of.cpu().numpy(), perm["row_of"])
    assert np.array_equal(L.src_of.cpu().numpy()[:rows], perm["src_of"])
    assert np.allclose(L.prob_perm.cpu().numpy()[:rows], fwd["prob_perm"], rtol=2e-6, atol=1e-7)
    # ---- bit-exact MX codes/scales of x ----
    ref_c, ref_s = mx.quantize_blocks(fwd["x_perm"], axis=1)
    assert np.array_equal(L.xq.cpu().numpy()[:rows], ref_c)
    assert np.array_equal(untile_scales(L.xq_s.cpu().numpy(), L.cap, wl.H)[:rows], ref_s)
    if training:
        ref_c, ref_s = mx.quantize_blocks(fwd["x_perm"], axis=0)
        assert np.array_equal(L.xq_col.cpu().numpy()[:, :rows], ref_c.T)
        assert np.array_equal(untile_scales(L.xq_col_s.cpu().numpy(), wl.H, L.cap)[:, :rows // 32], ref_s.T)
    # ---- forward floats ----
    assert_close(f64(L.y)[:rows], fwd["y"], "y")
    assert_close(f64(L.out), fwd["out"], "out")
    res = {"out_rel": rel_frob(f64(L.out), fwd["out"])}
    if training:
        gu = f64(L.saved_gu)[:rows]
        assert_close(gu[:, :wl.I], fwd["g"], "g")
        assert_close(gu[:, wl.I:], fwd["u"], "u")
        aq_col = mx.dequantize_blocks(L.aq_col.cpu().numpy()[:, :rows],
                                      untile_scales(L.aq_col_s.cpu().numpy(), wl.I, L.cap)[:, :rows // 32], axis=1)
        ref_aq_col = np.zeros((rows, wl.I))
        offs, split = perm["offsets_pad"], perm["split_sizes"]
        for e in range(wl.E):
            sl = slice(offs[e], offs[e] + split[e])
            ref_aq_col[sl] = ef.q_tokens(fwd["a"][sl], ef.MXFP8)
        assert_close(aq_col.T, ref_aq_col, "a quantized along tokens")
        assert_close(f64(L.dx), bwd["dx"], "dx")
        assert_close(f64(L.dwgu), bwd["dw_gu"], "dW_gu")
        assert_close(f64(L.dwd), bwd["dw_d"], "dW_d")
        assert_close(L.dprob.cpu().numpy(), bwd["dprob"], "dprob")
        res.update({k: rel_frob(f64(getattr(L, a)), bwd[b]) for k, a, b in
                    (("dx_rel", "dx", "dx"), ("dwgu_rel", "dwgu", "dw_gu"), ("dwd_rel", "dwd", "dw_d"))})
    if report is not None:
        report.update(res)
    return L, fwd, bwd


def test_tiny_workload_fwd_bwd():
    wl = configs.get(configs.TINY)
    check_layer(wl, synth.make_inputs(wl, 0), True)


@pytest.mark.parametrize("T,H,I,E,k,routing", [
    (300, 256, 384, 6, 2, "biased"),     # ragged segments, N tails in the backward GEMMs
    (200, 128, 128, 1, 1, "normal"),     # one expert: a plain GEMM
    (1000, 256, 256, 64, 6, "biased"),   # fine-grained, skewed, empty experts
    (513, 384, 640, 5, 3, "normal"),
    (600, 128, 128, 256, 8, "biased"),   # the largest E and k: 256 tiny segments, many empty
    (1, 128, 128, 4, 2, "normal"),       # one token
    (100, 128, 256, 4, 4, "normal"),     # k = E: every token in every expert
])
def test_small_workloads_fwd_bwd(T, H, I, E, k, routing):
    wl = configs.small(T, H, I, E, k, routing=routing, backward=True)
    check_layer(wl, synth.make_inputs(wl, 0), True)


def test_segment_sizes_around_tile_edges():
    """Experts with 1, 31, 32, 33, 127, 128, 129 and 0 tokens (k = 1)."""
    sizes = [1, 31, 32, 33, 127, 128, 129, 0]
    T = sum(sizes)
    wl = configs.small(T, 128, 256, len(sizes), 1, backward=True)
    inp = synth.make_inputs(wl, 0)
    owner = np.repeat(np.arange(len(sizes)), sizes)
    owner = np.random.default_rng(0).permutation(owner)
    logits = torch.zeros(T, len(sizes))
    logits[torch.arange(T), torch.from_numpy(owner)] = 5.0
    inp["logits"] = logits
    L, fwd, _ = check_layer(wl, inp, True)
    assert L.split_sizes.cpu().tolist() == sizes


def test_uneven_zipf_workload_forward():
    """The Zipf-loaded workload at full size, forward only (one expert empty)."""
    wl = configs.get(configs.UNEVEN)
    inp = synth.make_inputs(wl, 0)
    L, fwd, _ = check_layer(wl, inp, False)
    split = L.split_sizes.cpu().numpy()
    assert split[-1] == 0 and split[0] > split[1] > split[3]


def test_rerun_is_bit_identical():
    wl = configs.small(700, 256, 256, 8, 2, routing="biased", backward=True)
    inp = synth.make_inputs(wl, 0)
    a = run_gpu(wl, inp, True)
    outs = [t.clone() for t in (a.out, a.dx, a.dwgu, a.dwd, a.dprob)]
    a.forward(inp["logits"].cuda(), inp["x"].cuda())
    a.backward(inp["dout"].cuda())
    torch.cuda.synchronize()
    for before, after in zip(outs, (a.out, a.dx, a.dwgu, a.dwd, a.dprob)):
        assert torch.equal(before, after)


def test_tiles_never_mix_experts():
    """Expert 2's rows from the full grouped call equal a call that holds only expert 2's tokens."""
    wl = configs.small(600, 256, 256, 4, 1, backward=False)
    inp = synth.make_inputs(wl, 0)
    A = run_gpu(wl, inp, False)
    idx = A.idx.cpu().numpy()[:, 0]
    toks = np.nonzero(idx == 2)[0]
    sub = configs.small(len(toks), 256, 256, 4, 1, backward=False)
    inp2 = {"x": inp["x"][toks], "w_gu": inp["w_gu"], "w_d": inp["w_d"],
            "logits": torch.full((len(toks), 4), -1.0).index_fill_(1, torch.tensor([2]), 3.0)}
    Bc = run_gpu(sub, inp2, False)
    split = A.split_sizes.cpu().numpy()
    off = int(sum((s + 127) // 128 * 128 for s in split[:2]))
    assert torch.equal(A.y[off:off + len(toks)], Bc.y[:len(toks)])
    assert torch.equal(A.out[torch.from_numpy(toks).cuda()], Bc.out)


def test_quantization_error_against_unquantized_reference():
    """Reported, not a parity gate: MXFP8 vs a bf16 unquantized oracle on the tiny workload."""
    wl = configs.get(configs.TINY)
    inp = synth.make_inputs(wl, 0)
    L = run_gpu(wl, inp, True)
    idx, prob = rt.route_topk(inp["logits"].numpy(), wl.k)
    ref = ef.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]),
                     ef.UNQUANTIZED_BF16)
    err = rel_frob(f64(L.out), ref["out"])
    print(f"quantization error (rel Frobenius, out): {err:.4f}")
    assert err < 0.1


def test_per_expert_weight_tensors_give_the_stacked_results():
    """A training step with one weight tensor per expert (lists) is bit-identical to stacked weights."""
    wl = configs.small(500, 256, 384, 6, 2, routing="biased", backward=True)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    runs = []
    for as_list in (False, True):
        L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=True)
        w_gu = [w.clone() for w in inp["w_gu"]] if as_list else inp["w_gu"]
        w_d = [w.clone() for w in inp["w_d"]] if as_list else inp["w_d"]
        L.quantize_weights(w_gu, w_d)
        L.forward(inp["logits"], inp["x"])
        L.backward(inp["dout"])
        torch.cuda.synchronize()
        assert L.device_error() == (0, 0)
        runs.append([t.clone() for t in (L.out, L.dx, L.dwgu, L.dwd, L.dprob)])
    for a, b in zip(*runs):
        assert torch.equal(a, b)


def test_nvtx_ranges_change_nothing():
    wl = configs.small(300, 256, 384, 6, 2, routing="biased", backward=True)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    res = []
    for nvtx in (False, True):
        L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=True, nvtx=nvtx)
        L.step(inp["w_gu"], inp["w_d"], inp["logits"], inp["x"], inp["dout"])
        torch.cuda.synchronize()
        res.append([t.clone() for t in (L.out, L.dx, L.dwgu, L.dwd, L.dprob)])
    for a, b in zip(*res):
        assert torch.equal(a, b)

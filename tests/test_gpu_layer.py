"""GPU expert-FFN layer vs the oracle on the same seeded inputs.

Bit-exact: routing indices, split_sizes, the permutation, the MX codes and
scales of x and of dOut (both axes each).  Floats (y, saved g/u, a after
quantization along rows and along tokens, dH after quantization along rows
and along tokens, out, dx, dW_gu, dW_d, dprob): relative Frobenius error
<= 5e-3 and max abs error <= 2e-2 * max|ref|.  Device buffers are sliced to
the padded row count on the device before they reach numpy, and numpy
RuntimeWarnings (a NaN or an overflow in a cast) fail the test.
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

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("error::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_mx_codes(codes, scales, codes_t, scales_t, ref, cap, rows, name):
    """Codes and scales of a [cap][K] row-wise MX tensor (and, when given, of its
    along-token copy [K][cap]) equal the oracle quantizer's on ref [rows][K]."""
    K = ref.shape[1]
    ref_c, ref_s = mx.quantize_blocks(ref, axis=1)
    assert np.array_equal(codes.view(cap, K)[:rows].cpu().numpy(), ref_c), f"{name} row codes"
    assert np.array_equal(untile_scales(scales.cpu().numpy(), cap, K)[:rows], ref_s), f"{name} row scales"
    if codes_t is not None:
        # segments start on 128-row boundaries and are zero-padded: blocks of 32 rows of the
        # whole padded tensor are the blocks along tokens inside every segment
        ref_c, ref_s = mx.quantize_blocks(ref, axis=0)
        assert np.array_equal(codes_t.view(K, cap)[:, :rows].cpu().numpy(), ref_c.T), f"{name} token codes"
        assert np.array_equal(untile_scales(scales_t.cpu().numpy(), K, cap)[:, :rows // 32], ref_s.T), \
            f"{name} token scales"


def dequant_rows(codes, scales, cap, K, rows):
    return mx.dequantize_blocks(codes.view(cap, K)[:rows].cpu().numpy(),
                                untile_scales(scales.cpu().numpy(), cap, K)[:rows], axis=1)


def dequant_cols(codes_t, scales_t, cap, K, rows):
    """The along-token MX copy [K][cap], dequantized and transposed back to [rows][K]."""
    return mx.dequantize_blocks(codes_t.view(K, cap)[:, :rows].cpu().numpy(),
                                untile_scales(scales_t.cpu().numpy(), K, cap)[:, :rows // 32], axis=1).T


def q_tokens_segments(v, offs, split):
    out = np.zeros_like(v)
    for e in range(len(split)):
        sl = slice(offs[e], offs[e] + split[e])
        out[sl] = ef.q_tokens(v[sl], ef.MXFP8)
    return out


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
    assert np.array_equal(L.src_of[:rows].cpu().numpy(), perm["src_of"])
    assert np.allclose(L.prob_perm[:rows].cpu().numpy(), fwd["prob_perm"], rtol=2e-6, atol=1e-7)
    # ---- bit-exact MX codes/scales of x ----
    check_mx_codes(L.xq, L.xq_s, L.xq_col if training else None, L.xq_col_s if training else None,
                   fwd["x_perm"], L.cap, rows, "x")
    # ---- forward floats ----
    assert_close(f64(L.y[:rows]), fwd["y"], "y")
    assert_close(f64(L.out), fwd["out"], "out")
    a_rows = dequant_rows(L.workspace_tensor("a_codes"), L.workspace_tensor("a_scales"), L.cap, wl.I, rows)
    assert_close(a_rows, ef.q_rowwise(fwd["a"], ef.MXFP8), "a quantized along rows")
    res = {"out_rel": rel_frob(f64(L.out), fwd["out"])}
    if training:
        gu = f64(L.saved_gu[:rows])
        assert_close(gu[:, :wl.I], fwd["g"], "g")
        assert_close(gu[:, wl.I:], fwd["u"], "u")
        offs, split = perm["offsets_pad"], perm["split_sizes"]
        aq_col = dequant_cols(L.aq_col, L.aq_col_s, L.cap, wl.I, rows)
        assert_close(aq_col, q_tokens_segments(fwd["a"], offs, split), "a quantized along tokens")
        # ---- bit-exact MX codes/scales of dOut gathered to rows (both axes) ----
        check_mx_codes(L.workspace_tensor("dy_codes"), L.workspace_tensor("dy_scales"),
                       L.workspace_tensor("dy_col_codes"), L.workspace_tensor("dy_col_scales"),
                       bwd["dy_perm"], L.cap, rows, "dY")
        # ---- dH = [dg | du] after its quantizers (inputs differ by accumulation order: tolerance) ----
        dh_rows = dequant_rows(L.workspace_tensor("dh_codes"), L.workspace_tensor("dh_scales"), L.cap, 2 * wl.I,
                               rows)
        assert_close(dh_rows, ef.q_rowwise(bwd["dH"], ef.MXFP8), "dH quantized along rows")
        dh_col = dequant_cols(L.workspace_tensor("dh_col_codes"), L.workspace_tensor("dh_col_scales"), L.cap,
                              2 * wl.I, rows)
        assert_close(dh_col, q_tokens_segments(bwd["dH"], offs, split), "dH quantized along tokens")
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
    (256, 128, 4096, 4, 2, "normal"),    # 64 dprob partials per row: the reduce splits them over warps
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


@pytest.mark.parametrize("k", [2, 6])
def test_nan_logits_route_like_the_oracle(k):
    """NaN logits rank below every number (-inf included): rows with fewer numbers than k
    still select k distinct experts, identical to the oracle's choice; the permutation stays
    bit-exact; probabilities match, NaN where the oracle has NaN."""
    T, E = 300, 6
    wl = configs.small(T, 128, 128, E, k, backward=False)
    inp = synth.make_inputs(wl, 0)
    logits = inp["logits"].clone()
    rng = np.random.default_rng(5)
    logits[rng.choice(T, 40, replace=False), 2] = float("nan")               # one NaN
    rows = rng.choice(T, 20, replace=False)
    logits[rows[:10], :E - 1] = float("nan")                                 # one number left
    logits[rows[10:], :] = float("nan")                                      # all NaN
    logits[rows[10:15], 3] = float("-inf")                                   # -inf beats NaN
    logits[rng.choice(T, 10, replace=False), 4] = float("inf")
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=False)
    L.route(logits.cuda(), inp["x"].cuda())
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    with np.errstate(invalid="ignore"):                                  # NaN - NaN in the oracle's softmax
        idx, prob = rt.route_topk(logits.numpy(), k)
    assert np.array_equal(L.idx.cpu().numpy(), idx)
    got = L.prob.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(prob))
    fin = ~np.isnan(prob)
    assert np.allclose(got[fin], prob[fin], rtol=2e-6, atol=1e-7)
    perm = rt.permute(idx, E)
    assert np.array_equal(L.split_sizes.cpu().numpy(), perm["split_sizes"])
    assert np.array_equal(L.row_of.cpu().numpy(), perm["row_of"])
    assert np.array_equal(L.src_of[:perm["rows"]].cpu().numpy(), perm["src_of"])


def test_outputs_at_16_byte_offsets_give_the_same_results():
    """The GEMM epilogues store 32 bytes per lane when the output pointers are 32-byte aligned
    and 16 bytes otherwise; y and saved g,u at a 16-byte (not 32-byte) offset give the same
    values as 256-byte aligned ones."""
    from moe_expert_ffn_03_gb300 import binding as B
    wl = configs.small(300, 256, 384, 6, 2, routing="biased", backward=True)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    L = run_gpu(wl, inp, True)
    cap = L.cap
    y_off = torch.empty(cap * wl.H + 8, dtype=torch.bfloat16, device="cuda")[8:].view(cap, wl.H)
    gu_off = torch.empty(cap * 2 * wl.I + 8, dtype=torch.bfloat16, device="cuda")[8:].view(cap, 2 * wl.I)
    assert y_off.data_ptr() % 32 == 16 and gu_off.data_ptr() % 32 == 16
    B.grouped_mlp_fwd(L.d, L.xq, L.xq_s, L.split_sizes, L.prob_perm, L.wgu_q, L.wgu_s, L.wd_q, L.wd_s, y_off, gu_off,
                      L.aq_col, L.aq_col_s, L.ws)
    torch.cuda.synchronize()
    rows = L.padded_rows()
    assert torch.equal(y_off[:rows], L.y[:rows])
    assert torch.equal(gu_off[:rows], L.saved_gu[:rows])

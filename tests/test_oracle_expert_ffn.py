"""Pins of the oracle's expert FFN: textbook special cases, finite differences, invariants."""
import numpy as np
import pytest
import torch

from oracle import expert_ffn as ef
from oracle import mxfp8 as mx
from oracle import routing as rt


def make_case(T=16, H=32, I=64, E=4, k=2, seed=0, wstd=0.3):
    rng = np.random.default_rng(seed)
    x = mx.bf16(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w_gu = mx.bf16(rng.standard_normal((E, 2 * I, H)) * wstd)
    w_d = mx.bf16(rng.standard_normal((E, H, I)) * wstd)
    dout = mx.bf16(rng.standard_normal((T, H)))
    idx, prob = rt.route_topk(logits, k)
    return x, idx, prob.astype(np.float64), w_gu, w_d, dout


def torch_swiglu_mlp(x, w_g, w_u, w_d):
    """Textbook SwiGLU MLP y = W_d (silu(W_g x) * (W_u x)) in float64 torch."""
    X = torch.tensor(x, dtype=torch.float64)
    g = X @ torch.tensor(w_g, dtype=torch.float64).T
    u = X @ torch.tensor(w_u, dtype=torch.float64).T
    return (torch.nn.functional.silu(g) * u) @ torch.tensor(w_d, dtype=torch.float64).T


def test_single_expert_top1_is_plain_swiglu_mlp():
    x, _, _, w_gu, w_d, _ = make_case(T=24, E=1, k=1)
    idx = np.zeros((24, 1), dtype=np.int32)
    prob = np.ones((24, 1))
    f = ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT)
    I = w_gu.shape[1] // 2
    ref = torch_swiglu_mlp(x, w_gu[0, :I], w_gu[0, I:], w_d[0]).numpy()
    assert np.allclose(f["out"], ref, rtol=1e-12, atol=1e-12)


def test_quantized_single_expert_is_swiglu_on_dequantized_operands():
    """With quantizers on, E=1/k=1/p=1 is the textbook MLP on the MX-dequantized operands."""
    x, _, _, w_gu, w_d, _ = make_case(T=32, E=1, k=1)
    idx = np.zeros((32, 1), dtype=np.int32)
    f = ef.forward(x, idx, np.ones((32, 1)), w_gu, w_d, ef.MXFP8)
    I = w_gu.shape[1] // 2
    c, s = mx.quantize_blocks(x, axis=1)
    xd = mx.dequantize_blocks(c, s, axis=1)
    c, s = mx.quantize_blocks(w_gu[0], axis=1)
    wgud = mx.dequantize_blocks(c, s, axis=1)
    X = torch.tensor(xd)
    a = torch.nn.functional.silu(X @ torch.tensor(wgud[:I]).T) * (X @ torch.tensor(wgud[I:]).T)
    a = a.to(torch.float32).to(torch.float64).numpy()
    c, s = mx.quantize_blocks(a, axis=1)
    ad = mx.dequantize_blocks(c, s, axis=1)
    c, s = mx.quantize_blocks(w_d[0], axis=1)
    wdd = mx.dequantize_blocks(c, s, axis=1)
    ref = mx.bf16(ad @ wdd.T)
    # rows of the single expert are the tokens in order
    assert np.allclose(f["y"][:32], ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    assert np.allclose(f["out"], ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def test_grouped_equals_per_token_loop():
    """The grouped per-expert loop equals an HF-style loop over tokens and slots."""
    x, idx, prob, w_gu, w_d, _ = make_case(T=40, H=64, I=64, E=5, k=2, seed=3)
    f = ef.forward(x, idx, prob, w_gu, w_d, ef.MXFP8)
    wq = ef.quantize_weights(w_gu, w_d)
    out = np.zeros_like(f["out"])
    for t in range(x.shape[0]):
        acc = np.zeros(x.shape[1])
        for j in range(idx.shape[1]):
            e = idx[t, j]
            xq = ef.q_rowwise(x[t:t + 1], ef.MXFP8)
            acc += ef.expert_forward_rows(xq, prob[t:t + 1, j], wq["gu"][e], wq["d"][e])["y"][0]
        out[t] = mx.bf16(acc)
    assert np.allclose(out, f["out"], rtol=0, atol=1e-9 * np.abs(out).max())


def test_prob_in_swiglu_equals_weighted_combine():
    """Applying p in ScaledSwiGLU equals a p-weighted combine (the down GEMM is linear, bias-free)."""
    x, idx, prob, w_gu, w_d, _ = make_case(T=30, seed=4)
    f1 = ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT)
    f0 = ef.forward(x, idx, np.ones_like(prob), w_gu, w_d, ef.EXACT)
    out2 = ef.combine(f0["y"], f0["perm"]["row_of"], prob=prob, nm=ef.EXACT)
    assert np.allclose(f1["out"], out2, rtol=1e-12, atol=1e-13)


def loss(x, idx, prob, w_gu, w_d, dout):
    return float(np.sum(ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT)["out"] * dout))


def fd_errors(case, n_sample=40, h=1e-6, backward=ef.backward):
    x, idx, prob, w_gu, w_d, dout = case
    f = ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT)
    b = backward(f, dout, ef.EXACT)
    rng = np.random.default_rng(11)
    worst = 0.0
    targets = {"x": (x, b["dx"]), "w_gu": (w_gu, b["dw_gu"]), "w_d": (w_d, b["dw_d"]), "prob": (prob, b["dprob"])}
    for name, (arr, grad) in targets.items():
        flat_n = arr.size
        picks = rng.choice(flat_n, size=min(n_sample, flat_n), replace=False)
        for p in picks:
            i = np.unravel_index(p, arr.shape)
            args = {"x": x, "w_gu": w_gu, "w_d": w_d, "prob": prob}
            plus = arr.copy()
            plus[i] += h
            minus = arr.copy()
            minus[i] -= h
            args[name] = plus
            lp = loss(args["x"], idx, args["prob"], args["w_gu"], args["w_d"], dout)
            args[name] = minus
            lm = loss(args["x"], idx, args["prob"], args["w_gu"], args["w_d"], dout)
            num = (lp - lm) / (2 * h)
            scale = max(1.0, abs(num))
            worst = max(worst, abs(num - grad[i]) / scale)
    return worst


def test_backward_matches_central_finite_differences():
    case = make_case(T=16, H=32, I=64, E=4, k=2, seed=5)
    assert fd_errors(case) < 1e-6


def test_finite_differences_catch_planted_sign_error(monkeypatch):
    """Planting a dropped term in the SwiGLU derivative must fail the FD pin."""
    real = ef.swiglu_backward

    def wrong(dA, g, u, p):
        dg, du, dp = real(dA, g, u, p)
        s = ef.sigmoid(g)
        return dA * np.asarray(p)[:, None] * u * s, du, dp      # silu' without the g*s*(1-s) term
    monkeypatch.setattr(ef, "swiglu_backward", wrong)
    case = make_case(T=16, H=32, I=64, E=4, k=2, seed=5)
    assert fd_errors(case) > 1e-3


def test_finite_differences_catch_transposed_wgrad(monkeypatch):
    """A swapped gate/up half in dW_gu must fail the FD pin."""
    real = ef.backward

    def wrong(fwd, dout, nm=ef.MXFP8):
        b = real(fwd, dout, nm)
        I = fwd["I"]
        b["dw_gu"] = np.concatenate([b["dw_gu"][:, I:], b["dw_gu"][:, :I]], axis=1)
        return b
    case = make_case(T=16, H=32, I=64, E=4, k=2, seed=6)
    assert fd_errors(case, backward=wrong) > 1e-3


def test_wgrad_token_blocks_stay_inside_expert_segments():
    """Changing tokens routed only to other experts leaves an expert's quantized dW unchanged."""
    x, idx, prob, w_gu, w_d, dout = make_case(T=64, H=32, I=64, E=4, k=1, seed=9)
    f = ef.forward(x, idx, prob, w_gu, w_d)
    b = ef.backward(f, dout)
    t_other = np.nonzero(idx[:, 0] != 0)[0]
    x2 = x.copy()
    x2[t_other] *= 3.0
    dout2 = dout.copy()
    dout2[t_other] *= -2.0
    f2 = ef.forward(x2, idx, prob, w_gu, w_d)
    b2 = ef.backward(f2, dout2)
    assert np.array_equal(b["dw_gu"][0], b2["dw_gu"][0])
    assert np.array_equal(b["dw_d"][0], b2["dw_d"][0])
    assert not np.array_equal(b["dw_gu"][1:], b2["dw_gu"][1:])


def test_empty_expert_has_zero_weight_gradient():
    x, idx, prob, w_gu, w_d, dout = make_case(T=32, E=4, k=1, seed=10)
    idx = np.where(idx == 2, 1, idx).astype(np.int32)            # nobody picks expert 2
    f = ef.forward(x, idx, prob, w_gu, w_d)
    b = ef.backward(f, dout)
    assert f["perm"]["split_sizes"][2] == 0
    assert np.all(b["dw_gu"][2] == 0) and np.all(b["dw_d"][2] == 0)


def test_quantization_error_is_small_but_nonzero():
    x, idx, prob, w_gu, w_d, dout = make_case(T=64, H=64, I=128, E=4, k=2, seed=12, wstd=0.1)
    fq = ef.forward(x, idx, prob, w_gu, w_d, ef.MXFP8)
    fr = ef.forward(x, idx, prob, w_gu, w_d, ef.UNQUANTIZED_BF16)
    rel = np.linalg.norm(fq["out"] - fr["out"]) / np.linalg.norm(fr["out"])
    assert 1e-3 < rel < 0.15
    bq = ef.backward(fq, dout, ef.MXFP8)
    br = ef.backward(fr, dout, ef.UNQUANTIZED_BF16)
    for key in ("dx", "dw_gu", "dw_d", "dprob"):
        rel = np.linalg.norm(bq[key] - br[key]) / np.linalg.norm(br[key])
        assert rel < 0.2, key


def test_bf16_path_backward_is_the_exact_backward_up_to_bf16_rounding():
    """The BF16-path backward rounds every stored tensor to bf16 (dY, dH, a and x along
    either axis, g/u, the outputs) and nothing else: it lies within a few bf16 steps of
    the exact (finite-difference-pinned) backward, and differs from it."""
    rng = np.random.default_rng(21)
    T, H, I, E, k = 96, 64, 96, 4, 2
    x = mx.bf16(rng.standard_normal((T, H)))
    w_gu = mx.bf16(rng.standard_normal((E, 2 * I, H)) * 0.1)
    w_d = mx.bf16(rng.standard_normal((E, H, I)) * 0.1)
    dout = mx.bf16(rng.standard_normal((T, H)) * 0.01)
    idx, prob = rt.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
    prob = prob.astype(np.float64)
    b16 = ef.backward(ef.forward(x, idx, prob, w_gu, w_d, ef.BF16_PATH), dout, ef.BF16_PATH)
    ex = ef.backward(ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT), dout, ef.EXACT)
    for key in ("dx", "dw_gu", "dw_d", "dprob"):
        rel = np.linalg.norm(b16[key] - ex[key]) / np.linalg.norm(ex[key])
        assert 1e-5 < rel < 2e-2, (key, rel)
    # the along-token operands are rounded: dW_d sums products of bf16 dY and bf16 a
    assert np.array_equal(ef.q_tokens(b16["dH"], ef.BF16_PATH), mx.bf16(b16["dH"]))

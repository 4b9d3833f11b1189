"""Parity at the full workload sizes, in the launch configuration bench.py times.

The whole layer runs on the GPU; the oracle then recomputes, one by one,
sampled outputs it can afford on the host: complete routing and permutation
(bit-exact), the MX codes of x (bit-exact), whole rows of y / out / dx /
dprob for sampled tokens, and sampled entries of dW_gu and dW_d (each a
full reduction over an expert's tokens).  The per-row and per-column pieces
call the oracle's own primitives in the order its per-expert loop uses them.
"""
import numpy as np
import pytest
import torch

from helpers import MAX_ABS_FRAC, REL_FROB, rel_frob, untile_scales
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


def check_sample(got, ref, name):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rf = rel_frob(got, ref)
    ma = float(np.abs(got - ref).max())
    assert rf <= REL_FROB, f"{name}: rel Frobenius {rf:.3e}"
    assert ma <= MAX_ABS_FRAC * float(np.abs(ref).max()), f"{name}: max abs {ma:.3e}"


class ExpertCache:
    """Oracle-quantized (dequantized float64) weights of one expert at a time."""

    def __init__(self, w_gu, w_d):
        self.w_gu, self.w_d = w_gu, w_d
        self.e = None

    def get(self, e):
        if self.e != e:
            gu = self.w_gu[e].float().numpy().astype(np.float64)
            d = self.w_d[e].float().numpy().astype(np.float64)
            self.q = {"gu": ef.q_rowwise(gu, ef.MXFP8), "d": ef.q_rowwise(d, ef.MXFP8),
                      "guT": ef.q_rowwise(gu.T, ef.MXFP8), "dT": ef.q_rowwise(d.T, ef.MXFP8)}
            self.e = e
        return self.q


def run_full(name, training):
    wl = configs.get(name)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=training)
    L.quantize_weights(inp["w_gu"], inp["w_d"])
    L.forward(inp["logits"], inp["x"])
    if training:
        L.backward(inp["dout"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    cpu = {k: v.cpu() for k, v in inp.items()}
    return wl, L, cpu


def check_routing_and_codes(wl, L, cpu):
    idx, prob = rt.route_topk(cpu["logits"].numpy(), wl.k)
    assert np.array_equal(L.idx.cpu().numpy(), idx)
    assert np.allclose(L.prob.cpu().numpy(), prob, rtol=2e-6, atol=1e-7)
    perm = rt.permute(idx, wl.E)
    rows = perm["rows"]
    assert np.array_equal(L.split_sizes.cpu().numpy(), perm["split_sizes"])
    assert np.array_equal(L.row_of.cpu().numpy(), perm["row_of"])
    assert np.array_equal(L.src_of.cpu().numpy()[:rows], perm["src_of"])
    # MX codes of every token row (quantize-then-gather equals gather-then-quantize)
    x = f64(cpu["x"])
    c, s = mx.quantize_blocks(x, axis=1)
    src = perm["src_of"]
    valid = src >= 0
    xq = L.xq.cpu().numpy()[:rows]
    assert np.array_equal(xq[valid], c[src[valid]])
    assert np.all(xq[~valid] == 0)
    xs = untile_scales(L.xq_s.cpu().numpy(), L.cap, wl.H)[:rows]
    assert np.array_equal(xs[valid], s[src[valid]])
    return idx, prob, perm


def sample_tokens(idx, experts, n, rng):
    ok = np.nonzero(np.all(np.isin(idx, experts), axis=1))[0]
    pick = list(ok[:2]) + list(ok[-2:]) + list(rng.choice(ok, size=min(n, len(ok)), replace=False))
    return sorted(set(int(t) for t in pick))


def check_rows(wl, L, cpu, idx, prob, perm, tokens, training):
    cache = ExpertCache(cpu["w_gu"], cpu["w_d"])
    x = cpu["x"]
    dout = cpu.get("dout")
    got_out, ref_out, got_dx, ref_dx, got_dp, ref_dp, got_y, ref_y = [], [], [], [], [], [], [], []
    per_e = {}
    for t in tokens:
        for j in range(wl.k):
            per_e.setdefault(int(idx[t, j]), []).append((t, j))
    y_rows, dx_rows, dp_vals = {}, {}, {}
    for e in sorted(per_e):
        q = cache.get(e)
        for t, j in per_e[e]:
            xr = ef.q_rowwise(x[t:t + 1].float().numpy().astype(np.float64), ef.MXFP8)
            p = np.array([float(prob[t, j])])
            f = ef.expert_forward_rows(xr, p, q["gu"], q["d"], ef.MXFP8)
            y_rows[(t, j)] = f["y"][0]
            if training:
                dyr = ef.q_rowwise(dout[t:t + 1].float().numpy().astype(np.float64), ef.MXFP8)
                dA = dyr @ q["dT"].T
                dg, du, dp = ef.swiglu_backward(dA, f["g"], f["u"], p)
                dH = mx.fp32(np.concatenate([dg, du], axis=1))
                dx_rows[(t, j)] = mx.bf16(ef.q_rowwise(dH, ef.MXFP8) @ q["guT"].T)[0]
                dp_vals[(t, j)] = float(mx.fp32(dp)[0])
    y_gpu = L.y
    for t in tokens:
        ref_out.append(mx.bf16(sum(y_rows[(t, j)] for j in range(wl.k))))
        got_out.append(f64(L.out[t]))
        for j in range(wl.k):
            got_y.append(f64(y_gpu[int(perm["row_of"][t, j])]))
            ref_y.append(y_rows[(t, j)])
        if training:
            ref_dx.append(mx.bf16(sum(dx_rows[(t, j)] for j in range(wl.k))))
            got_dx.append(f64(L.dx[t]))
            ref_dp.append([dp_vals[(t, j)] for j in range(wl.k)])
            got_dp.append(L.dprob[t].cpu().numpy())
    check_sample(got_y, ref_y, "y rows")
    check_sample(got_out, ref_out, "out rows")
    if training:
        check_sample(got_dx, ref_dx, "dx rows")
        check_sample(got_dp, ref_dp, "dprob")


def check_wgrad_entries(wl, L, cpu, prob, perm, experts, rng, n=4):
    """Sampled dW_d[e][h][i] and dW_gu[e][j][h]: full token reductions per expert."""
    cache = ExpertCache(cpu["w_gu"], cpu["w_d"])
    offs, split, src = perm["offsets_pad"], perm["split_sizes"], perm["src_of"]
    prob_perm = np.zeros(perm["rows"])
    prob_perm[perm["row_of"].ravel()] = prob.ravel()
    I, H = wl.I, wl.H
    got_d, ref_d, got_g, ref_g = [], [], [], []
    for e in experts:
        m = int(split[e])
        if m == 0:
            assert torch.count_nonzero(L.dwd[e]) == 0 and torch.count_nonzero(L.dwgu[e]) == 0
            continue
        q = cache.get(e)
        toks = src[offs[e]:offs[e] + m]
        xq_rows = ef.q_rowwise(cpu["x"][toks].float().numpy().astype(np.float64), ef.MXFP8)
        dyq_rows = ef.q_rowwise(cpu["dout"][toks].float().numpy().astype(np.float64), ef.MXFP8)
        p = prob_perm[offs[e]:offs[e] + m][:, None]
        hs = rng.choice(H, size=n, replace=False)
        cols_i = rng.choice(I, size=n, replace=False)
        for h, i in zip(hs, cols_i):
            g = xq_rows @ q["gu"][i]
            u = xq_rows @ q["gu"][I + i]
            a = mx.fp32(ef.silu(g) * u * p[:, 0])
            dy = cpu["dout"][toks, h].float().numpy().astype(np.float64)
            ref_d.append(float(ef.q_tokens(dy[:, None], ef.MXFP8)[:, 0] @ ef.q_tokens(a[:, None], ef.MXFP8)[:, 0]))
            got_d.append(float(L.dwd[e, h, i]))
            # dW_gu rows j = i (gate) and I + i (up) at column h
            dA = dyq_rows @ q["dT"][i]
            dg, du, _ = ef.swiglu_backward(dA[:, None], mx.bf16(g)[:, None], mx.bf16(u)[:, None], p[:, 0])
            xc = cpu["x"][toks, h].float().numpy().astype(np.float64)
            xcq = ef.q_tokens(xc[:, None], ef.MXFP8)[:, 0]
            for jj, col in ((i, dg), (I + i, du)):
                ref_g.append(float(ef.q_tokens(mx.fp32(col), ef.MXFP8)[:, 0] @ xcq))
                got_g.append(float(L.dwgu[e, jj, h]))
    check_sample(got_d, ref_d, "dW_d entries")
    check_sample(got_g, ref_g, "dW_gu entries")


def test_mixtral_fwd_bwd_full_size():
    wl, L, cpu = run_full(configs.MIXTRAL_FWDBWD, True)
    idx, prob, perm = check_routing_and_codes(wl, L, cpu)
    rng = np.random.default_rng(0)
    experts = sorted(set(int(e) for e in idx[0]))
    toks = sample_tokens(idx, experts, 4, rng)
    check_rows(wl, L, cpu, idx, prob, perm, toks, True)
    check_wgrad_entries(wl, L, cpu, prob, perm, experts[:1], rng, n=3)


def test_mixtral_forward_full_size():
    wl, L, cpu = run_full(configs.MIXTRAL_FWD, False)
    idx, prob, perm = check_routing_and_codes(wl, L, cpu)
    rng = np.random.default_rng(1)
    experts = sorted(set(int(e) for e in idx[-1]))
    check_rows(wl, L, cpu, idx, prob, perm, sample_tokens(idx, experts, 4, rng), False)


def test_finegrained_fwd_bwd_full_size():
    wl, L, cpu = run_full(configs.FINEGRAINED, True)
    idx, prob, perm = check_routing_and_codes(wl, L, cpu)
    split = perm["split_sizes"]
    assert np.count_nonzero(split == 0) >= 1, "expected at least one empty expert"
    rng = np.random.default_rng(2)
    toks = sorted(set([0, wl.T - 1] + list(rng.choice(wl.T, 10, replace=False))))
    check_rows(wl, L, cpu, idx, prob, perm, toks, True)
    busiest = int(np.argmax(split))
    empty = int(np.nonzero(split == 0)[0][0])
    light = int(np.nonzero(split > 0)[0][np.argmin(split[split > 0])])
    check_wgrad_entries(wl, L, cpu, prob, perm, [busiest, light, empty], rng, n=4)

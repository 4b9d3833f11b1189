"""Parity at the full workload sizes, in the launch configuration bench.py times.

The whole layer runs on the GPU; the oracle then recomputes, one by one,
sampled outputs it can afford on the host: complete routing and permutation
(bit-exact), the MX codes of x (bit-exact), whole rows of y / out / dx /
dprob for sampled tokens, and one entry of dW_gu and of dW_d in every
256 x 256 output tile of the busiest expert, of an expert whose token range
is an odd number of 128-row blocks, and (fine-grained) of the lightest and an
empty expert -- each entry a full reduction over the expert's tokens.  The
per-row and per-column pieces call the oracle's own primitives in the order
its per-expert loop uses them.
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


def check_wgrad_tiles(wl, L, cpu, prob, perm, experts, rng):
    """One entry of dW_d[e] ([H][I]) and one of dW_gu[e] ([2I][H]) in EVERY 256 x 256 output
    tile of each listed expert, each a full reduction over the expert's tokens, recomputed
    with the oracle's primitives in its per-expert order (the columns of a and dH that the
    sampled entries need are computed as batched matmuls of the same operands).  An expert
    without tokens must have all-zero gradients."""
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
        p = prob_perm[offs[e]:offs[e] + m]
        # dW_d tiles (hb, ib): entry (h, i); dW_gu tiles (jb, hb): entry (j, h), j < I gate, j >= I up
        def pick(n, blk):                                 # an index inside 256-block blk of range(n)
            return blk * 256 + int(rng.integers(min(256, n - blk * 256)))

        d_ent = [(pick(H, hb), pick(I, ib)) for hb in range(-(-H // 256)) for ib in range(-(-I // 256))]
        g_ent = [(pick(2 * I, jb), pick(H, hb)) for jb in range(-(-2 * I // 256)) for hb in range(-(-H // 256))]
        cols = sorted(set(i for _, i in d_ent) | set(j % I for j, _ in g_ent))
        ci = {c: n for n, c in enumerate(cols)}
        cols = np.array(cols)
        g = xq_rows @ q["gu"][cols].T                     # [m][n] gate columns
        u = xq_rows @ q["gu"][I + cols].T                 # [m][n] up columns
        a = mx.fp32(ef.silu(g) * u * p[:, None])          # the quantizer input of a
        a_tok = ef.q_tokens(a, ef.MXFP8)
        dA = dyq_rows @ q["dT"][cols].T                   # [m][n]
        dg, du, _ = ef.swiglu_backward(dA, mx.bf16(g), mx.bf16(u), p)
        dg_tok = ef.q_tokens(mx.fp32(dg), ef.MXFP8)
        du_tok = ef.q_tokens(mx.fp32(du), ef.MXFP8)
        h_d = np.array([h for h, _ in d_ent])
        dy_tok = ef.q_tokens(cpu["dout"][toks][:, h_d].float().numpy().astype(np.float64), ef.MXFP8)
        h_g = np.array([h for _, h in g_ent])
        x_tok = ef.q_tokens(cpu["x"][toks][:, h_g].float().numpy().astype(np.float64), ef.MXFP8)
        dwd_e = L.dwd[e].float().cpu().numpy()
        dwgu_e = L.dwgu[e].float().cpu().numpy()
        for n, (h, i) in enumerate(d_ent):
            ref_d.append(float(dy_tok[:, n] @ a_tok[:, ci[i]]))
            got_d.append(float(dwd_e[h, i]))
        for n, (j, h) in enumerate(g_ent):
            col = (dg_tok if j < I else du_tok)[:, ci[j % I]]
            ref_g.append(float(col @ x_tok[:, n]))
            got_g.append(float(dwgu_e[j, h]))
    check_sample(got_d, ref_d, "dW_d entries (one per 256 x 256 tile)")
    check_sample(got_g, ref_g, "dW_gu entries (one per 256 x 256 tile)")


def odd_block_expert(split, exclude):
    """An expert (other than `exclude`) whose padded token range is an odd number of
    128-row blocks: its weight-gradient tiles end in a short barrier stage."""
    for e in np.argsort(-split, kind="stable"):
        nb = -(-int(split[e]) // 128)
        if int(e) not in exclude and nb % 2 == 1:
            return [int(e)]
    return []


def test_mixtral_fwd_bwd_full_size():
    wl, L, cpu = run_full(configs.MIXTRAL_FWDBWD, True)
    idx, prob, perm = check_routing_and_codes(wl, L, cpu)
    rng = np.random.default_rng(0)
    experts = sorted(set(int(e) for e in idx[0]))
    toks = sample_tokens(idx, experts, 12, rng)
    check_rows(wl, L, cpu, idx, prob, perm, toks, True)
    split = perm["split_sizes"]
    busiest = int(np.argmax(split))
    check_wgrad_tiles(wl, L, cpu, prob, perm, [busiest] + odd_block_expert(split, {busiest}), rng)


def test_mixtral_forward_full_size():
    wl, L, cpu = run_full(configs.MIXTRAL_FWD, False)
    idx, prob, perm = check_routing_and_codes(wl, L, cpu)
    rng = np.random.default_rng(1)
    experts = sorted(set(int(e) for e in idx[-1]))
    check_rows(wl, L, cpu, idx, prob, perm, sample_tokens(idx, experts, 12, rng), False)


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
    chosen = [busiest, light, empty]
    check_wgrad_tiles(wl, L, cpu, prob, perm, chosen + odd_block_expert(split, set(chosen)), rng)

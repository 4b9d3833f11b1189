"""Routing and permutation on both of its GPU paths, against the oracle.

Up to E * ceil(T/32) <= 16384 mask words, top-k and the per-expert scan are one launch
(the block that finishes last scans); above that the scan has a kernel of its own.
Either way the permutation is finished by the launch that quantizes the x rows.  Both
paths must give the oracle's idx, split_sizes, row_of and src_of bit for bit, zero the
padding rows (src_of = -1, prob_perm = 0, x codes and scale codes 0), and give each
token the same probabilities whichever path routed it.  The outputs are filled with
garbage first, so that nothing passes by being zero already; the route-only entry point
(moe_route) is checked the same way, and repeated calls on one workspace (the block
ticket must return to zero) stay identical.
"""
import numpy as np
import pytest
import torch

from helpers import untile_scales
from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN, route_launches
from oracle import mxfp8 as mx
from oracle import routing as rt

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("error::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def route(T, H, E, k, routing="normal", seed=0, logits=None, renorm=True):
    wl = configs.small(T, H, 128, E, k, routing=routing, backward=False)
    inp = synth.make_inputs(wl, seed)
    if logits is not None:
        inp["logits"] = logits
    L = ExpertFFN(T, H, 128, E, k, training=False, renormalize=renorm)
    for buf, v in ((L.src_of, 0x5A5A5A5A), (L.row_of, 0x5A5A5A5A), (L.idx, 0x5A5A5A5A)):
        buf.fill_(v)
    L.prob_perm.fill_(3.0)
    L.xq.fill_(0x7F)
    L.xq_s.fill_(0x7F)
    L.route(inp["logits"].cuda(), inp["x"].cuda())
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    return L, inp


def check_against_oracle(L, inp, T, H, E, k, renorm=True):
    idx, prob = rt.route_topk(inp["logits"].numpy(), k, renormalize=renorm)
    perm = rt.permute(idx, E)
    rows, offs, split = perm["rows"], perm["offsets_pad"], perm["split_sizes"]
    assert np.array_equal(L.idx.cpu().numpy(), idx)
    # a softmax over all E divides by an f32 sum of E exponentials: a looser bound
    assert np.allclose(L.prob.cpu().numpy(), prob, rtol=2e-6 if renorm else 1e-5, atol=1e-7)
    assert np.array_equal(L.split_sizes.cpu().numpy(), split)
    assert np.array_equal(L.row_of.cpu().numpy(), perm["row_of"])
    src_of = L.src_of[:rows].cpu().numpy()
    assert np.array_equal(src_of, perm["src_of"])
    pp = L.prob_perm[:rows].cpu().numpy()
    pad = perm["src_of"] < 0
    assert np.all(pp[pad] == 0.0)
    real = ~pad
    # every real row carries the probability of the (token, slot) that maps to it
    flat_rows = perm["row_of"].reshape(-1)
    got_prob = L.prob.cpu().numpy().reshape(-1)
    assert np.array_equal(pp[flat_rows], got_prob)
    # x codes: the oracle quantizer on the gathered rows, zero codes and scales in padding rows
    x = inp["x"].float().numpy().astype(np.float64)
    x_perm = np.zeros((rows, H))
    x_perm[real] = x[perm["src_of"][real]]
    ref_c, ref_s = mx.quantize_blocks(x_perm, axis=1)
    codes = L.xq.view(L.cap, H)[:rows].cpu().numpy()
    scales = untile_scales(L.xq_s.cpu().numpy(), L.cap, H)[:rows]
    assert np.array_equal(codes, ref_c)
    assert np.array_equal(scales, ref_s)
    assert np.count_nonzero(codes[pad]) == 0 and np.count_nonzero(scales[pad]) == 0
    for e in range(E):
        assert offs[e] % 128 == 0
    return prob


@pytest.mark.parametrize("T,E,k,routing,path", [
    (65536, 8, 2, "biased", 1),     # E * ceil(T/32) = 16384 mask words: the fused bound, inclusive
    (65537, 8, 2, "biased", 2),     # one 32-token group past it
    (2048, 256, 1, "normal", 1),    # 256 experts, 16384 words
    (2049, 256, 8, "normal", 2),    # one group past it, k = 8
    (1000, 7, 3, "normal", 1),      # ragged T, E not a multiple of 4 (scalar logit loads)
    (41000, 13, 3, "normal", 2),    # the same on the two-launch path (13 * 1282 words)
    (1, 4, 2, "normal", 1),         # a single token
    (33, 4, 4, "normal", 1),        # k = E, a second group of one token
])
def test_route_paths_match_the_oracle(T, E, k, routing, path):
    assert route_launches(T, E) == path
    H = 128
    L, inp = route(T, H, E, k, routing)
    check_against_oracle(L, inp, T, H, E, k)


@pytest.mark.parametrize("T,E,k,renorm", [
    (9000, 64, 6, True),            # 64 x 282 groups > 16384 words: two launches, four lanes per token
    (9000, 64, 6, False),           # softmax over all 64 experts
    (15000, 37, 3, False),          # E not a multiple of 4 on the four-lane top-k
])
def test_many_experts_two_launch_path(T, E, k, renorm):
    assert route_launches(T, E) == 2
    H = 128
    L, inp = route(T, H, E, k, "biased", renorm=renorm)
    check_against_oracle(L, inp, T, H, E, k, renorm)


def test_both_paths_route_each_token_alike():
    """The first 65536 tokens routed alone (one launch) and inside 65600 tokens (two):
    the same experts and bit-identical probabilities."""
    E, k, H = 8, 2, 128
    big, inp = route(65600, H, E, k, "biased", seed=3)
    small, _ = route(65536, H, E, k, "biased", seed=3, logits=inp["logits"][:65536].clone())
    assert route_launches(65600, E) == 2 and route_launches(65536, E) == 1
    assert torch.equal(big.idx[:65536], small.idx)
    assert torch.equal(big.prob[:65536], small.prob)


@pytest.mark.parametrize("T,E,k", [(4096, 8, 2), (70000, 8, 2)])
def test_route_only_entry_and_repeated_calls(T, E, k):
    """moe_route (maps without quantized rows) equals the oracle, and five calls in a row
    on one workspace give identical results on both paths."""
    H = 128
    wl = configs.small(T, H, 128, E, k, routing="biased", backward=False)
    inp = synth.make_inputs(wl, 2)
    L = ExpertFFN(T, H, 128, E, k, training=False)
    logits = inp["logits"].cuda()
    first = None
    for _ in range(5):
        for buf in (L.src_of, L.row_of, L.idx, L.split_sizes):
            buf.fill_(0x5A5A5A5A)
        L.prob_perm.fill_(3.0)
        B.moe_route(L.d, logits, L.idx, L.prob, L.split_sizes, L.row_of, L.src_of, L.prob_perm, L.ws)
        torch.cuda.synchronize()
        assert L.device_error() == (0, 0)
        got = [t.clone() for t in (L.idx, L.prob, L.split_sizes, L.row_of, L.src_of, L.prob_perm)]
        if first is None:
            first = got
        assert all(torch.equal(a, b) for a, b in zip(first, got))
    idx, prob = rt.route_topk(inp["logits"].numpy(), k)
    perm = rt.permute(idx, E)
    rows = perm["rows"]
    assert np.array_equal(L.idx.cpu().numpy(), idx)
    assert np.array_equal(L.split_sizes.cpu().numpy(), perm["split_sizes"])
    assert np.array_equal(L.row_of.cpu().numpy(), perm["row_of"])
    assert np.array_equal(L.src_of[:rows].cpu().numpy(), perm["src_of"])
    pp = L.prob_perm[:rows].cpu().numpy()
    assert np.all(pp[perm["src_of"] < 0] == 0.0)
    assert np.array_equal(pp[perm["row_of"].reshape(-1)], L.prob.cpu().numpy().reshape(-1))


def test_expert_without_tokens_on_the_single_cta_path():
    """Experts that no token picks get empty segments (no padding rows either)."""
    T, E, k, H = 640, 6, 2, 128
    wl = configs.small(T, H, 128, E, k, backward=False)
    logits = synth.make_inputs(wl, 1)["logits"].clone()
    logits[:, 1] = -1e30
    logits[:, 4] = -1e30
    L, inp = route(T, H, E, k, logits=logits)
    split = L.split_sizes.cpu().numpy()
    assert split[1] == 0 and split[4] == 0 and split.sum() == T * k
    check_against_oracle(L, inp, T, H, E, k)

"""The sampled full-size checks, run against the complete oracle on a small
workload: row- and entry-wise recomputation must agree with the per-expert loop."""
import numpy as np
import torch

import test_gpu_fullsize as fs
from helpers import tile_scales
from moe_expert_ffn_03_gb300 import configs, synth
from oracle import expert_ffn as ef
from oracle import mxfp8 as mx
from oracle import routing as rt


class OracleLayer:
    """Holds the full oracle results in the attribute layout of the device layer."""

    def __init__(self, wl, inp):
        f64 = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
        idx, prob = rt.route_topk(inp["logits"].numpy(), wl.k)
        fwd = ef.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]))
        bwd = ef.backward(fwd, f64(inp["dout"]))
        perm = fwd["perm"]
        self.cap = perm["rows"] + 128
        bf = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)  # noqa: E731
        self.idx = torch.from_numpy(idx)
        self.prob = torch.from_numpy(prob)
        self.split_sizes = torch.from_numpy(perm["split_sizes"])
        self.row_of = torch.from_numpy(perm["row_of"])
        src = np.full(self.cap, -1, np.int32)
        src[:perm["rows"]] = perm["src_of"]
        self.src_of = torch.from_numpy(src)
        xp = np.zeros((self.cap, wl.H))
        xp[:perm["rows"]] = fwd["x_perm"]
        c, s = mx.quantize_blocks(xp, axis=1)
        self.xq = torch.from_numpy(c)
        self.xq_s = torch.from_numpy(tile_scales(s))
        y = np.zeros((self.cap, wl.H))
        y[:perm["rows"]] = fwd["y"]
        self.y = bf(y)
        self.out = bf(fwd["out"])
        self.dx = bf(bwd["dx"])
        self.dprob = torch.from_numpy(bwd["dprob"].astype(np.float32))
        self.dwd = bf(bwd["dw_d"])
        self.dwgu = bf(bwd["dw_gu"])


def test_sampled_checks_agree_with_full_oracle():
    wl = configs.small(400, 384, 384, 6, 2, routing="biased", backward=True)   # partial 256-tiles on both axes
    inp = synth.make_inputs(wl, 0)
    L = OracleLayer(wl, inp)
    idx, prob, perm = fs.check_routing_and_codes(wl, L, inp)
    rng = np.random.default_rng(0)
    experts = sorted(set(int(e) for e in idx[0]))
    fs.check_rows(wl, L, inp, idx, prob, perm, fs.sample_tokens(idx, experts, 5, rng), True)
    split = perm["split_sizes"]
    assert fs.odd_block_expert(split, set()), "the workload should hold an odd-block expert"
    fs.check_wgrad_tiles(wl, L, inp, prob, perm, list(range(wl.E)), rng)


def test_sampled_wgrad_check_catches_a_wrong_tile():
    """A single wrong dW entry in one 256 x 256 tile fails the per-tile check."""
    import pytest
    wl = configs.small(300, 384, 384, 4, 2, routing="biased", backward=True)
    inp = synth.make_inputs(wl, 0)
    L = OracleLayer(wl, inp)
    idx, prob, perm = fs.check_routing_and_codes(wl, L, inp)
    e = int(np.argmax(perm["split_sizes"]))
    # corrupt the whole last (partial) tile of dW_gu[e]: whichever entry the check samples
    L.dwgu[e, 512:, 256:] = -L.dwgu[e, 512:, 256:] * 3
    with pytest.raises(AssertionError):
        fs.check_wgrad_tiles(wl, L, inp, prob, perm, [e], np.random.default_rng(0))

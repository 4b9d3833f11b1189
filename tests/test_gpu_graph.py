"""A step captured as a CUDA graph replays the eager step's results bit for bit, also after
its input tensors are refilled in place."""
import pytest
import torch

from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _eager(wl, training, inp):
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=training)
    L.step(inp["w_gu"], inp["w_d"], inp["logits"], inp["x"], inp.get("dout"))
    torch.cuda.synchronize()
    return [t.clone() for t in ((L.out, L.dx, L.dwgu, L.dwd, L.dprob) if training else (L.out,))]


@pytest.mark.parametrize("training", [True, False])
def test_graph_replay_equals_eager_step(training):
    wl = configs.small(500, 256, 384, 6, 2, routing="biased", backward=training)
    a = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    b = {k: v.cuda() for k, v in synth.make_inputs(wl, 1).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=training)
    static = {k: v.clone() for k, v in a.items()}
    g = L.capture_step(static["w_gu"], static["w_d"], static["logits"], static["x"], static.get("dout"))
    for inp in (b, a, b):
        for k in static:
            static[k].copy_(inp[k])
        g.replay()
        torch.cuda.synchronize()
        assert L.device_error() == (0, 0)
        got = (L.out, L.dx, L.dwgu, L.dwd, L.dprob) if training else (L.out,)
        for x, y in zip(got, _eager(wl, training, inp)):
            assert torch.equal(x, y)

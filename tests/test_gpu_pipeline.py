"""Host-fed steps with overlapped copies give the serial path's results bit for bit."""
import pytest
import torch

from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN
from moe_expert_ffn_03_gb300.pipeline import HostPipeline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


@pytest.mark.parametrize("training", [True, False])
def test_pipelined_steps_equal_serial_steps(training):
    wl = configs.small(600, 256, 384, 6, 2, routing="biased", backward=training)
    weights = synth.make_inputs(wl, 0, with_grad=False)
    w_gu, w_d = weights["w_gu"].cuda(), weights["w_d"].cuda()
    names = ("x", "logits", "dout") if training else ("x", "logits")
    steps = [synth.make_inputs(wl, seed, with_grad=training) for seed in (1, 2, 3, 4)]
    host_in = [{n: st[n].pin_memory() for n in names} for st in steps]

    ref = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=training)
    expect = []
    for st in steps:
        ref.quantize_weights(w_gu, w_d)
        ref.forward(st["logits"].cuda(), st["x"].cuda())
        res = {"out": ref.out.clone()}
        if training:
            ref.backward(st["dout"].cuda())
            res["dx"] = ref.dx.clone()
        expect.append({k: v.cpu() for k, v in res.items()})

    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=training)
    pipe = HostPipeline(L, w_gu, w_d)
    outs = [{"out": torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory(),
             "dx": torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()} for _ in steps]
    pipe.run(host_in[:2], outs[:2])
    pipe.run(host_in[2:], outs[2:])          # a second call reuses the slots and events
    pipe.join()
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    for got, exp in zip(outs, expect):
        assert torch.equal(got["out"], exp["out"])
        if training:
            assert torch.equal(got["dx"], exp["dx"])

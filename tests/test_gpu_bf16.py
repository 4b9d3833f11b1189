"""BF16 grouped forward (no quantization) vs the oracle with the bf16-activation numerics."""
import numpy as np
import pytest
import torch

from helpers import assert_close
from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN
from oracle import expert_ffn as ef
from oracle import routing as rt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name_or_dims", [
    configs.TINY,
    (300, 256, 384, 6, 2, "biased"),
    (513, 384, 640, 5, 3, "normal"),
    configs.UNEVEN,
])
def test_bf16_forward_matches_oracle(name_or_dims):
    wl = configs.get(name_or_dims) if isinstance(name_or_dims, str) else configs.small(*name_or_dims[:5],
                                                                                         routing=name_or_dims[5])
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0, with_grad=False).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=False)
    L.route(inp["logits"], inp["x"])
    out = L.forward_bf16(inp["x"], inp["w_gu"], inp["w_d"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    idx, prob = rt.route_topk(inp["logits"].cpu().numpy(), wl.k)
    fwd = ef.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]), ef.BF16_PATH)
    rows = fwd["perm"]["rows"]
    assert np.array_equal(f64(L.x_perm)[:rows], fwd["x_perm"])
    assert_close(f64(L.a_perm)[:rows], ef.q_rowwise(fwd["a"], ef.BF16_PATH), "a (bf16)")
    assert_close(f64(L.y_b16)[:rows], fwd["y"], "y")
    assert_close(f64(out), fwd["out"], "out")

"""Device-side failure detection without a fault: a GEMM launch whose producer issues
no loads has every consumer wait run out; the kernel reports MOE_ERR_DEVICE_TIMEOUT,
returns, and the context keeps working."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_reports_and_context_survives():
    build.build()
    scratch = torch.zeros(96 * 1024, dtype=torch.uint8, device="cuda")
    code, site = B.moe_selftest_wait_timeout(scratch, 20_000_000)       # 20 ms limit
    assert code == 6, (code, site)                                        # MOE_ERR_DEVICE_TIMEOUT
    assert 500 <= site < 600
    # a normal layer step afterwards still runs and reports no error
    wl = configs.get(configs.TINY)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=True)
    L.quantize_weights(inp["w_gu"], inp["w_d"])
    out = L.forward(inp["logits"], inp["x"]).float().cpu().numpy()
    L.backward(inp["dout"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    assert np.all(np.isfinite(out)) and np.abs(out).max() > 0

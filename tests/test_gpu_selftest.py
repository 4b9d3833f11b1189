"""The MXFP8 MMA issue self-test (the tensor pipe's ceiling for the GEMM's
instruction mix) runs cleanly, reports one CTA pair per two SMs, and its rate
is of the order the tensor cores allow: a sanity check, not a benchmark."""
import pytest
import torch

from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build

pytestmark = pytest.mark.gpu


def test_mma_issue_selftest_runs_and_reports():
    build.build()
    scratch = torch.zeros(256, dtype=torch.uint8, device="cuda")
    k_steps = 4096
    B.moe_selftest_mma_issue(64, scratch)                         # warm-up
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    pairs = B.moe_selftest_mma_issue(k_steps, scratch)
    e1.record()
    torch.cuda.synchronize()
    assert B.moe_get_device_error(scratch) == (0, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert pairs == sms // 2
    tflops = pairs * k_steps * 2.0 * 256 * 256 * 128 / (e0.elapsed_time(e1) * 1e-3) / 1e12
    print(f"MXFP8 MMA issue rate: {tflops:.0f} TFLOP/s over {pairs} pairs")
    assert 500.0 < tflops < 20000.0

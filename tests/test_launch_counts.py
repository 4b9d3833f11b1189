"""Host logic of the launch counts that bench.py reports as gpu_launches.

Routing is one launch while the per-expert token masks hold at most 16384 words
(E * ceil(T/32)), two past that; the permutation is finished by the row quantizer.  The
Python rule must match the bound the CUDA source uses to pick the one-launch path.
"""
import os
import re

from moe_expert_ffn_03_gb300 import configs
from moe_expert_ffn_03_gb300.layer import ROUTE_SCAN_FUSED_MAX_WORDS, launches_per_step, route_launches

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_route_bound_matches_the_cuda_source():
    src = open(os.path.join(ROOT, "moe_expert_ffn_03_gb300", "csrc", "route_permute.cu")).read()
    m = re.search(r"constexpr int RS_SCAN_MAX_WORDS = (\d+);", src)
    assert m is not None
    assert int(m.group(1)) == ROUTE_SCAN_FUSED_MAX_WORDS


def test_route_launches_at_the_bound():
    assert route_launches(65536, 8) == 1          # 8 x 2048 = 16384 words
    assert route_launches(65537, 8) == 2
    assert route_launches(2048, 256) == 1
    assert route_launches(2049, 256) == 2
    assert route_launches(1, 4) == 1


def test_launches_per_step_of_the_workloads():
    # uneven Zipf forward: weights 2, routing 1, permutation + rows 1, GEMMs 2, combine 1
    wl = configs.get("uneven_zipf_T4096_H1024_I2816_E8_k2")
    assert launches_per_step(wl.T, wl.E, wl.k, wl.backward) == 7
    # Mixtral-shaped training: one-launch routing (4096 mask words), 16 launches
    wl = configs.get("mixtral_fwdbwd_T16384_H4096_I14336_E8_k2")
    assert launches_per_step(wl.T, wl.E, wl.k, wl.backward) == 16
    # fine-grained training: 65536 mask words, two-launch routing, 17 launches
    wl = configs.get("finegrained_T32768_H2048_I1408_E64_k6")
    assert launches_per_step(wl.T, wl.E, wl.k, wl.backward) == 17

"""The five expert-FFN workloads (sizes, routing structure, pass).

T tokens, H hidden, I intermediate (gate_up has 2*I outputs), E experts,
k experts per token.  ``backward`` says whether the workload runs the
backward pass.  Every workload uses seed 0 and synthetic inputs from
``synth.make_inputs``.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    routing: str          # "normal" | "zipf" | "biased"
    backward: bool
    zipf_s: float = 1.2
    bias_std: float = 2.0
    w_std: float = 0.02
    g_std: float = 0.01

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops_fwd(self) -> float:
        """Algorithmic forward FLOPs of the two grouped GEMMs: 2*R*H*2I + 2*R*I*H."""
        return 6.0 * self.R * self.H * self.I

    def flops_total(self) -> float:
        """Forward, plus dgrad and wgrad of both GEMMs when the workload trains."""
        return (18.0 if self.backward else 6.0) * self.R * self.H * self.I


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_T256_H128_I256_E4_k2", 256, 128, 256, 4, 2, "normal", True),
        Workload("uneven_zipf_T4096_H1024_I2816_E8_k2", 4096, 1024, 2816, 8, 2, "zipf", False),
        Workload("mixtral_fwd_T16384_H4096_I14336_E8_k2", 16384, 4096, 14336, 8, 2, "normal", False),
        Workload("mixtral_fwdbwd_T16384_H4096_I14336_E8_k2", 16384, 4096, 14336, 8, 2, "normal", True),
        Workload("finegrained_T32768_H2048_I1408_E64_k6", 32768, 2048, 1408, 64, 6, "biased", True),
    )
}

ORDER = list(WORKLOADS)          # index 0..4 in the order above
TINY, UNEVEN, MIXTRAL_FWD, MIXTRAL_FWDBWD, FINEGRAINED = ORDER


def get(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[ORDER[name_or_index]]
    return WORKLOADS[name_or_index]


def small(T: int, H: int, I: int, E: int, k: int, routing: str = "normal", backward: bool = True,
          name: str | None = None) -> Workload:
    """An ad-hoc workload for parity tests (same distributions as the named ones)."""
    return Workload(name or f"small_T{T}_H{H}_I{I}_E{E}_k{k}_{routing}", T, H, I, E, k, routing, backward)

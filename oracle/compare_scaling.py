"""Accuracy of MX block scaling against per-tensor FP8 scaling (oracle only).

[BioNeMo-MoE], section "MoE训练的瓶颈与TE的对应能力": FP8 and MXFP8 differ in
the granularity of the scale, and the finer MX granularity is there to keep
range and precision.  This script measures what that buys on the expert FFN
forward: the relative Frobenius error of the combined output (and of the
activation a) of each numerics against the exact forward (float64, no
rounding, no quantizers), on the seeded synthetic workloads:

  * MXFP8              -- one power-of-two scale per 32 values (the product path)
  * per-tensor FP8     -- one dynamic scale per expert operand tensor
  * BF16 activations   -- no quantization, bf16 between the GEMMs

Test infrastructure: it imports only the oracle and the input generator.

    python -m oracle.compare_scaling [--tokens-finegrained 4096]
"""
from __future__ import annotations

import argparse
import time

import numpy as np

from . import expert_ffn as ef
from . import fp8_tensor as pt
from .routing import route_topk


def _forward_weights_mx(w_gu, w_d):
    """The two forward weight operands of the MXFP8 oracle, quantized expert by expert."""
    return {"gu": np.stack([ef.q_rowwise(w, ef.MXFP8) for w in w_gu]),
            "d": np.stack([ef.q_rowwise(w, ef.MXFP8) for w in w_d])}


def rel_fro(a, ref) -> float:
    return float(np.linalg.norm(np.asarray(a) - ref) / np.linalg.norm(ref))


def compare(x, logits, w_gu, w_d, k: int) -> dict:
    """Errors of the three numerics against the exact forward on one input set."""
    idx, prob = route_topk(np.asarray(logits, dtype=np.float32), k)
    prob = prob.astype(np.float64)
    exact = ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT)
    rows = {"mxfp8": ef.forward(x, idx, prob, w_gu, w_d, ef.MXFP8, wq=_forward_weights_mx(w_gu, w_d)),
            "fp8_per_tensor": pt.forward(x, idx, prob, w_gu, w_d),
            "bf16_activations": ef.forward(x, idx, prob, w_gu, w_d, ef.BF16_PATH)}
    out = {}
    ref = exact["out"]
    ref_norm = np.linalg.norm(ref, axis=1)
    live = ref_norm > 0
    for name, f in rows.items():
        tok = np.linalg.norm(f["out"] - ref, axis=1)[live] / ref_norm[live]
        out[name] = {"out_rel_fro": rel_fro(f["out"], ref),
                     "out_token_rel_mean": float(np.mean(tok)),   # every token weighs the same
                     "out_token_rel_max": float(np.max(tok)),
                     "a_rel_fro": rel_fro(f["a"], exact["a"])}   # a as it enters its quantizer
    split = exact["perm"]["split_sizes"]
    out["loads"] = {"min": int(split.min()), "max": int(split.max()), "empty": int((split == 0).sum())}
    return out


def workload_inputs(wl, tokens: int | None = None):
    """Float64 views of a workload's seeded inputs (first `tokens` tokens if given)."""
    import dataclasses

    from moe_expert_ffn_03_gb300 import synth
    if tokens is not None and tokens < wl.T:
        wl = dataclasses.replace(wl, T=tokens, name=f"{wl.name}_first{tokens}")
    d = synth.make_inputs(wl, 0, with_grad=False)
    f = {k: v.double().numpy() for k, v in d.items()}
    return wl, f["x"], f["logits"], f["w_gu"], f["w_d"]


def with_outlier_channels(x, every: int = 128, factor: float = 100.0):
    """Stress variant (not a workload of the pages): every `every`-th hidden channel of x
    scaled by `factor` and rounded back to bf16 -- a few large channels inside every
    token, the case where one scale per tensor wastes range."""
    from .mxfp8 import bf16
    y = np.array(x, dtype=np.float64)
    y[:, ::every] *= factor
    return bf16(y)


def with_outlier_tokens(x, every: int = 16, factor: float = 4096.0):
    """Stress variant (not a workload of the pages): every `every`-th token of x scaled by
    `factor` (a power of two: exact in bf16) -- tokens of very different magnitude sharing
    one expert's per-tensor scale."""
    y = np.array(x, dtype=np.float64)
    y[::every] *= factor
    return y


def main():
    from moe_expert_ffn_03_gb300 import configs
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens-finegrained", type=int, default=4096)
    args = ap.parse_args()
    variants = (("", lambda x: x),
                ("  + outlier channels (x[:, ::128] * 100)", with_outlier_channels),
                ("  + outlier tokens (x[::16] * 4096)", with_outlier_tokens))
    for name, tokens in ((configs.UNEVEN, None), (configs.FINEGRAINED, args.tokens_finegrained)):
        for label, make in variants:
            t0 = time.time()
            wl, x, logits, w_gu, w_d = workload_inputs(configs.get(name), tokens)
            r = compare(make(x), logits, w_gu, w_d, wl.k)
            print(f"{wl.name}{label}  (loads min {r['loads']['min']} max {r['loads']['max']} "
                  f"empty {r['loads']['empty']}; {time.time() - t0:.0f} s)")
            for key in ("mxfp8", "fp8_per_tensor", "bf16_activations"):
                v = r[key]
                print(f"    {key:18s} out rel-Fro {v['out_rel_fro']:.3e}  per-token mean {v['out_token_rel_mean']:.3e}"
                      f"  per-token max {v['out_token_rel_max']:.3e}  a rel-Fro {v['a_rel_fro']:.3e}")


if __name__ == "__main__":
    main()

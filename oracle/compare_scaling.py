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


def _weights_mx(w_gu, w_d, backward: bool):
    """The weight operands of the MXFP8 oracle, quantized expert by expert (the two
    forward ones, and the two transposed ones of the backward when asked)."""
    wq = {"gu": np.stack([ef.q_rowwise(w, ef.MXFP8) for w in w_gu]),
          "d": np.stack([ef.q_rowwise(w, ef.MXFP8) for w in w_d])}
    if backward:
        wq["guT"] = np.stack([ef.q_rowwise(w.T, ef.MXFP8) for w in w_gu])
        wq["dT"] = np.stack([ef.q_rowwise(w.T, ef.MXFP8) for w in w_d])
    return wq


def _token_rel(got, ref):
    """Mean over tokens of |got_t - ref_t| / |ref_t| (tokens with a zero reference skipped)."""
    n = np.linalg.norm(ref, axis=1)
    live = n > 0
    return np.linalg.norm(got - ref, axis=1)[live] / n[live]


def rel_fro(a, ref) -> float:
    return float(np.linalg.norm(np.asarray(a) - ref) / np.linalg.norm(ref))


def _weights_bf16(w_gu, w_d):
    """The BF16 path's weight operands: the bf16 master weights as they are (rounding bf16
    values to bf16 changes nothing), the transposed ones as views -- no copies."""
    return {"gu": w_gu, "d": w_d, "guT": np.swapaxes(w_gu, 1, 2), "dT": np.swapaxes(w_d, 1, 2)}


def compare(x, logits, w_gu, w_d, k: int, dout=None) -> dict:
    """Errors of the three numerics against the exact forward (and, given dout, the
    exact backward) on one input set.  One numerics at a time, keeping only its
    errors, so the largest workloads fit in host memory."""
    idx, prob = route_topk(np.asarray(logits, dtype=np.float32), k)
    prob = prob.astype(np.float64)
    train = dout is not None
    exact = ef.forward(x, idx, prob, w_gu, w_d, ef.EXACT)
    ref_out, ref_a = exact["out"], exact["a"]
    exb = ef.backward(exact, dout, ef.EXACT) if train else None
    split = exact["perm"]["split_sizes"]
    del exact
    runs = {
        "mxfp8": (lambda: ef.forward(x, idx, prob, w_gu, w_d, ef.MXFP8, wq=_weights_mx(w_gu, w_d, train)),
                  lambda f: ef.backward(f, dout, ef.MXFP8)),
        "fp8_per_tensor": (lambda: pt.forward(x, idx, prob, w_gu, w_d),
                           lambda f: pt.backward(f, dout)),
        "bf16_activations": (lambda: ef.forward(x, idx, prob, w_gu, w_d, ef.BF16_PATH, wq=_weights_bf16(w_gu, w_d)),
                             lambda f: ef.backward(f, dout, ef.BF16_PATH)),
    }
    out = {}
    for name, (fwd_fn, bwd_fn) in runs.items():
        f = fwd_fn()
        tok = _token_rel(f["out"], ref_out)
        out[name] = {"out_rel_fro": rel_fro(f["out"], ref_out),
                     "out_token_rel_mean": float(np.mean(tok)),   # every token weighs the same
                     "out_token_rel_max": float(np.max(tok)),
                     "a_rel_fro": rel_fro(f["a"], ref_a)}        # a as it enters its quantizer
        if train:
            g = bwd_fn(f)
            tok = _token_rel(g["dx"], exb["dx"])
            out[name].update({"dx_rel_fro": rel_fro(g["dx"], exb["dx"]),
                              "dx_token_rel_mean": float(np.mean(tok)),
                              "dw_gu_rel_fro": rel_fro(g["dw_gu"], exb["dw_gu"]),
                              "dw_d_rel_fro": rel_fro(g["dw_d"], exb["dw_d"]),
                              "dprob_rel_fro": rel_fro(g["dprob"], exb["dprob"])})
            del g
        del f
    out["loads"] = {"min": int(split.min()), "max": int(split.max()), "empty": int((split == 0).sum())}
    return out


def workload_inputs(wl, tokens: int | None = None):
    """Float64 views of a workload's seeded inputs (first `tokens` tokens if given); the
    upstream gradient dout is drawn for every workload, also the forward-only ones."""
    import dataclasses

    from moe_expert_ffn_03_gb300 import synth
    if tokens is not None and tokens < wl.T:
        wl = dataclasses.replace(wl, T=tokens, name=f"{wl.name}_first{tokens}")
    d = synth.make_inputs(wl, 0, with_grad=True)
    f = {k: v.double().numpy() for k, v in d.items()}
    return wl, f["x"], f["logits"], f["w_gu"], f["w_d"], f["dout"]


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
    ap.add_argument("--workloads", default="uneven,finegrained", help="comma-separated: uneven, finegrained")
    args = ap.parse_args()
    chosen = set(args.workloads.split(","))
    variants = (("", lambda x: x),
                ("  + outlier channels (x[:, ::128] * 100)", with_outlier_channels),
                ("  + outlier tokens (x[::16] * 4096)", with_outlier_tokens))
    table = (("uneven", configs.UNEVEN, None), ("finegrained", configs.FINEGRAINED, args.tokens_finegrained))
    for key, name, tokens in table:
        if key not in chosen:
            continue
        for label, make in variants:
            t0 = time.time()
            wl, x, logits, w_gu, w_d, dout = workload_inputs(configs.get(name), tokens)
            r = compare(make(x), logits, w_gu, w_d, wl.k, dout)
            print(f"{wl.name}{label}  (loads min {r['loads']['min']} max {r['loads']['max']} "
                  f"empty {r['loads']['empty']}; {time.time() - t0:.0f} s)")
            for num in ("mxfp8", "fp8_per_tensor", "bf16_activations"):
                v = r[num]
                print(f"    {num:18s} out rel-Fro {v['out_rel_fro']:.3e}  per-token mean {v['out_token_rel_mean']:.3e}"
                      f"  per-token max {v['out_token_rel_max']:.3e}  a rel-Fro {v['a_rel_fro']:.3e}")
                print(f"    {'':18s} dx rel-Fro {v['dx_rel_fro']:.3e}  per-token mean {v['dx_token_rel_mean']:.3e}"
                      f"  dW_gu {v['dw_gu_rel_fro']:.3e}  dW_d {v['dw_d_rel_fro']:.3e}"
                      f"  dprob {v['dprob_rel_fro']:.3e}", flush=True)


if __name__ == "__main__":
    main()

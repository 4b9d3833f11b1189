"""Per-tensor FP8 with dynamic scaling: the oracle's forward and backward (test infrastructure only).

[英伟达开源MoE加速神器], section "3. Transformer Engine：FP8 训练加速": the Hopper
FP8 recipe keeps 8-bit training usable through dynamic scaling of each tensor.
[BioNeMo-MoE], sections "MoE训练的瓶颈与TE的对应能力" and "MXFP8与融合MLP": FP8
and MXFP8 differ in the granularity of the scale -- MXFP8 gives every 32
consecutive values their own scale, FP8 one scale per tensor.

Readings (listed in the design notes):
* Element format E4M3, as for MXFP8, for every tensor including the
  gradients, so a comparison with MXFP8 isolates the granularity of the scale
  (the pages name no other format for either path).
* Dynamic scaling = the scale follows the tensor's own current amax:
  s = fp32(448 / amax) with amax = max |v| over the tensor (s = 1 when the
  tensor is all zero); code = RNE_E4M3(fp32(v * s)), saturating to +-448;
  value = code / s.  Tensors holding NaN or Inf are outside this path.
* The tensors are the operands of each expert's GEMMs, as the grouped call
  keeps them: expert e's token rows of x (its split by split_sizes), its own
  weights W_gu[e] and W_d[e], and its rows of the activation a.  So every
  operand carries one scale per expert.
* The activation a = silu(g) * u * p is stored as bf16 before it is quantized:
  a per-tensor scale needs the whole tensor's amax before any element can be
  quantized, so the intermediate is materialized (the unfused path).
* The GEMMs accumulate exactly here (float64 on dequantized operands); the
  output y is rounded to bf16 and combined as in the MXFP8 path.
"""
from __future__ import annotations

import numpy as np

from . import mxfp8 as mx
from .expert_ffn import combine, silu, swiglu_backward
from .routing import permute

E4M3_MAX = np.float32(448.0)


def tensor_scale(amax) -> float:
    """s = fp32(448 / amax) (1 for an all-zero tensor), a float32 value."""
    a = np.float32(amax)
    if not np.isfinite(a):
        raise ValueError("per-tensor FP8: the tensor holds NaN or Inf")
    if a == 0:
        return 1.0
    return float(E4M3_MAX / a)


def quantize_tensor(v):
    """(codes uint8 with v's shape, scale s) of one tensor."""
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    amax = float(np.max(np.abs(v32))) if v32.size else 0.0
    s = tensor_scale(amax)
    y = (v32 * np.float32(s)).astype(np.float64)     # the float32 product
    return mx.e4m3_encode(y), s


def dequantize_tensor(codes, s) -> np.ndarray:
    return mx.e4m3_decode(codes) / np.float64(s)


def qdq(v):
    """Quantize-dequantize one tensor; returns (values, s)."""
    c, s = quantize_tensor(v)
    return dequantize_tensor(c, s), s


def quantize_weights(w_gu, w_d):
    """Per-expert codes and scales of the two forward weight operands."""
    E = np.shape(w_gu)[0]
    out = {"gu": [], "gu_s": np.zeros(E), "d": [], "d_s": np.zeros(E)}
    for e in range(E):
        c, s = quantize_tensor(w_gu[e])
        out["gu"].append(c)
        out["gu_s"][e] = s
        c, s = quantize_tensor(w_d[e])
        out["d"].append(c)
        out["d_s"][e] = s
    out["gu"] = np.stack(out["gu"])
    out["d"] = np.stack(out["d"])
    return out


def forward(x, idx, prob, w_gu, w_d, wq=None):
    """Forward of the expert FFN with per-tensor FP8 operands.

    x [T][H], idx/prob [T][k] from route_topk, w_gu [E][2I][H], w_d [E][H][I].
    Per expert e (rows of its segment, in the expert-major order):
      xq = Q(x_e)            one scale s_x[e]
      g|u = xq @ Q(W_gu[e])^T
      a = bf16(fp32(silu(g) * u * p))
      y = bf16(Q(a) @ Q(W_d[e])^T)    scales s_a[e], s_d[e]
    then out[t] = sum_j y[row_of[t][j]].
    """
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    E, twoI, _ = np.shape(w_gu)
    I = twoI // 2
    perm = permute(idx, E)
    rows, src_of, offs = perm["rows"], perm["src_of"], perm["offsets_pad"]
    split = perm["split_sizes"]
    if wq is None:
        wq = quantize_weights(w_gu, w_d)
    prob = np.asarray(prob, dtype=np.float64)
    prob_perm = np.zeros(rows)
    prob_perm[perm["row_of"].ravel()] = prob.ravel()
    valid = src_of >= 0
    x_perm = np.zeros((rows, H))
    x_perm[valid] = x[src_of[valid]]
    xq_codes = np.zeros((rows, H), dtype=np.uint8)
    aq_codes = np.zeros((rows, I), dtype=np.uint8)
    a = np.zeros((rows, I))
    g_all = np.zeros((rows, I))
    u_all = np.zeros((rows, I))
    y = np.zeros((rows, H))
    s_x = np.ones(E)
    s_a = np.ones(E)
    for e in range(E):                               # the per-expert loop
        r0, m = int(offs[e]), int(split[e])
        if m == 0:
            continue
        sl = slice(r0, r0 + m)
        cx, s_x[e] = quantize_tensor(x_perm[sl])
        xq_codes[sl] = cx
        wgu = dequantize_tensor(wq["gu"][e], wq["gu_s"][e])
        gu = dequantize_tensor(cx, s_x[e]) @ wgu.T
        g, u = gu[:, :I], gu[:, I:]
        g_all[sl], u_all[sl] = mx.bf16(g), mx.bf16(u)
        a[sl] = mx.bf16(mx.fp32(silu(g) * u * prob_perm[sl][:, None]))
        ca, s_a[e] = quantize_tensor(a[sl])
        aq_codes[sl] = ca
        wd = dequantize_tensor(wq["d"][e], wq["d_s"][e])
        y[sl] = mx.bf16(dequantize_tensor(ca, s_a[e]) @ wd.T)
    out = combine(y, perm["row_of"])
    return {"perm": perm, "prob_perm": prob_perm, "x_perm": x_perm, "xq_codes": xq_codes, "s_x": s_x,
            "g": g_all, "u": u_all, "a": a, "aq_codes": aq_codes, "s_a": s_a, "y": y, "out": out, "wq": wq,
            "I": I}


def backward(fwd, dout):
    """Backward of ``forward`` with straight-through per-tensor quantizers.

    One scale per expert operand tensor, as in the forward: expert e's rows of
    dY (= dout gathered) and of dH = [dg | du], its weights (the forward's codes,
    read transposed) and its rows of x and a (the forward's codes).  A per-tensor
    scale does not depend on the axis, so the dgrad and the wgrad GEMMs consume
    the same codes.  g and u are kept in bf16 from the forward; dH is stored in
    bf16 before its quantization (its scale needs the tensor's amax).
    """
    perm, wq = fwd["perm"], fwd["wq"]
    dout = np.asarray(dout, dtype=np.float64)
    T, H = dout.shape
    I = fwd["I"]
    E = len(perm["split_sizes"])
    rows, src_of, offs = perm["rows"], perm["src_of"], perm["offsets_pad"]
    split = perm["split_sizes"]
    valid = src_of >= 0
    dy_perm = np.zeros((rows, H))
    dy_perm[valid] = dout[src_of[valid]]
    dx_perm = np.zeros((rows, H))
    dp_perm = np.zeros(rows)
    dw_gu = np.zeros((E, 2 * I, H))
    dw_d = np.zeros((E, H, I))
    for e in range(E):                               # the per-expert loop
        r0, m = int(offs[e]), int(split[e])
        if m == 0:
            continue
        sl = slice(r0, r0 + m)
        dyq, _ = qdq(dy_perm[sl])
        wd = dequantize_tensor(wq["d"][e], wq["d_s"][e])        # [H][I]
        wgu = dequantize_tensor(wq["gu"][e], wq["gu_s"][e])     # [2I][H]
        dA = dyq @ wd                                            # [m][I]
        g, u = fwd["g"][sl], fwd["u"][sl]
        dg, du, dp = swiglu_backward(dA, g, u, fwd["prob_perm"][sl])
        dH = mx.bf16(mx.fp32(np.concatenate([dg, du], axis=1)))
        dhq, _ = qdq(dH)
        dp_perm[sl] = dp
        aq = dequantize_tensor(fwd["aq_codes"][sl], fwd["s_a"][e])
        xq = dequantize_tensor(fwd["xq_codes"][sl], fwd["s_x"][e])
        dw_d[e] = dyq.T @ aq
        dx_perm[sl] = dhq @ wgu
        dw_gu[e] = dhq.T @ xq
    dx_perm = mx.bf16(dx_perm)
    dx = combine(dx_perm, perm["row_of"])
    return {"dx": dx, "dw_gu": mx.bf16(dw_gu), "dw_d": mx.bf16(dw_d),
            "dprob": mx.fp32(dp_perm[perm["row_of"]]), "dp_perm": dp_perm}

"""Per-expert loop forward and backward of the oracle (test infrastructure only).

[BioNeMo-MoE], section "GroupedLinear": the baseline runs one Python loop
iteration (one GEMM launch) per expert; the grouped form applies every
expert's own weight to that expert's tokens, selected by split_sizes, with
gate_up out_features = 2 * intermediate_size and bias=False.  Section
"MXFP8与融合MLP": gate_up -> ScaledSwiGLU (SwiGLU times the router
probability) -> down, with MXFP8 quantization before every GEMM and 16-bit
master weights; the fused op has a matching backward.

This module IS the per-expert loop: ``for e in range(E)`` with one dense
float64 matmul per expert.  Every product of two dequantized MXFP8 values is
exact and float64 accumulation bounds the oracle's own summation error far
below the float32 accumulation of the device path.

Readings (listed in the design notes):
* W_gu[e] rows 0..I-1 are the gate, rows I..2I-1 the up projection;
  a = silu(g) * u * p with silu(g) = g / (1 + exp(-g)).
* p is applied once, in ScaledSwiGLU; the combine is a plain sum over the k
  slots (fp32-exact sum of bf16 values, rounded to bf16).
* Every MX block runs along the contraction axis of the GEMM that consumes
  the tensor: x, a, dY, dH rowwise for the dgrad/forward GEMMs; x, a, dY, dH
  along tokens (inside each expert segment) for the wgrad GEMMs; W_gu and W_d
  along H resp. I for the forward and along 2I resp. H for the backward.
* Backward quantizers are straight-through: the backward GEMMs consume MX
  copies quantized along their own contraction axis; g and u are saved as
  bf16 and read back by the backward.
* The bf16 outputs (y, out, dX, dW) are float32 results rounded to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import mxfp8 as mx
from .routing import permute


@dataclass(frozen=True)
class Numerics:
    """quantized: MXFP8 quantizers on (False = identity quantizers).
    rounded: float32 quantizer inputs, bf16 saved g/u and bf16 outputs
    (False = pure float64, used by the finite-difference checks).
    act_bf16: with quantizers off, every tensor a GEMM consumes is rounded to
    bf16 instead, along either axis (the BF16 path of the recipe stores its
    activations and gradients in bf16)."""
    quantized: bool = True
    rounded: bool = True
    act_bf16: bool = False


MXFP8 = Numerics(True, True)
UNQUANTIZED_BF16 = Numerics(False, True)
BF16_PATH = Numerics(False, True, True)
EXACT = Numerics(False, False)


def silu(g):
    return g / (1.0 + np.exp(-g))


def sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


def _f32(v, nm: Numerics):
    return mx.fp32(v) if nm.rounded else np.asarray(v, dtype=np.float64)


def _bf16(v, nm: Numerics):
    return mx.bf16(v) if nm.rounded else np.asarray(v, dtype=np.float64)


def q_rowwise(v, nm: Numerics):
    """Quantize-dequantize along the last axis (identity when quantizers are off)."""
    if not nm.quantized:
        return mx.bf16(v) if nm.act_bf16 else np.asarray(v, dtype=np.float64)
    c, s = mx.quantize_blocks(v, axis=-1)
    return mx.dequantize_blocks(c, s, axis=-1)


def q_tokens(v, nm: Numerics):
    """Quantize-dequantize one expert's rows along the token axis (axis 0).

    Blocks of 32 consecutive rows start at the first row of the expert's
    segment; a partial last block is padded with zero rows.  With quantizers
    off: the identity, or bf16 rounding in the BF16 path.
    """
    v = np.asarray(v, dtype=np.float64)
    if not nm.quantized:
        return mx.bf16(v) if nm.act_bf16 else v
    if v.shape[0] == 0:
        return v
    m = v.shape[0]
    mp = -(-m // mx.BLOCK) * mx.BLOCK
    pad = np.zeros((mp,) + v.shape[1:])
    pad[:m] = v
    c, s = mx.quantize_blocks(pad, axis=0)
    return mx.dequantize_blocks(c, s, axis=0)[:m]


def quantize_weights(w_gu, w_d, nm: Numerics = MXFP8):
    """Dequantized views of the four weight operands (per expert, float64).

    gu  : W_gu[e] [2I][H] blocks along H   (forward gate_up B operand)
    d   : W_d[e]  [H][I]  blocks along I   (forward down B operand)
    guT : W_gu[e]^T [H][2I] blocks along 2I (gate_up dgrad B operand)
    dT  : W_d[e]^T  [I][H]  blocks along H  (down dgrad B operand)
    """
    w_gu = np.asarray(w_gu, dtype=np.float64)
    w_d = np.asarray(w_d, dtype=np.float64)
    return {
        "gu": q_rowwise(w_gu, nm),
        "d": q_rowwise(w_d, nm),
        "guT": q_rowwise(np.swapaxes(w_gu, 1, 2), nm),
        "dT": q_rowwise(np.swapaxes(w_d, 1, 2), nm),
    }


def expert_forward_rows(xq_rows, p_rows, wq_gu_e, wq_d_e, nm: Numerics = MXFP8):
    """Forward of ONE expert on some of its (already quantized) rows.

    xq_rows [m][H] dequantized MX rows of x, p_rows [m] router probabilities.
    Returns dict g, u (as saved for the backward), a (the float32 quantizer
    input), aq (a after the rowwise quantizer) and y [m][H] (bf16 output).
    Only rowwise quantizers act here, so any subset of rows gives the same
    values as the full segment.
    """
    I = wq_gu_e.shape[0] // 2
    gu = xq_rows @ wq_gu_e.T                        # [m][2I]
    g, u = gu[:, :I], gu[:, I:]
    a = _f32(silu(g) * u * np.asarray(p_rows, dtype=np.float64)[:, None], nm)
    aq = q_rowwise(a, nm)
    y = _bf16(aq @ wq_d_e.T, nm)                    # [m][H]
    return {"g": _bf16(g, nm), "u": _bf16(u, nm), "a": a, "aq": aq, "y": y}


def forward(x, idx, prob, w_gu, w_d, nm: Numerics = MXFP8, wq=None):
    """Whole forward: permute, quantize x, per-expert loop, combine.

    x [T][H], idx/prob [T][k] from route_topk, w_gu [E][2I][H], w_d [E][H][I].
    Returns the permutation, the permuted-row tensors (rows = padded row
    count; padding rows are zero) and out [T][H].
    """
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    E, twoI, _ = np.shape(w_gu)
    I = twoI // 2
    k = np.shape(idx)[1]
    perm = permute(idx, E)
    rows, src_of, offs = perm["rows"], perm["src_of"], perm["offsets_pad"]
    split = perm["split_sizes"]
    if wq is None:
        wq = quantize_weights(w_gu, w_d, nm)
    prob = np.asarray(prob, dtype=np.float64)
    prob_perm = np.zeros(rows)
    valid = src_of >= 0
    flat_row = perm["row_of"].ravel()
    prob_perm[flat_row] = prob.ravel()
    x_perm = np.zeros((rows, H))
    x_perm[valid] = x[src_of[valid]]
    xq_perm = q_rowwise(x_perm, nm)                  # gather, then quantize rows
    g = np.zeros((rows, I))
    u = np.zeros((rows, I))
    a = np.zeros((rows, I))
    y = np.zeros((rows, H))
    for e in range(E):                               # the per-expert loop
        r0, m = int(offs[e]), int(split[e])
        if m == 0:
            continue
        sl = slice(r0, r0 + m)
        f = expert_forward_rows(xq_perm[sl], prob_perm[sl], wq["gu"][e], wq["d"][e], nm)
        g[sl], u[sl], a[sl], y[sl] = f["g"], f["u"], f["a"], f["y"]
    out = combine(y, perm["row_of"], nm=nm)
    return {"perm": perm, "prob_perm": prob_perm, "x_perm": x_perm, "xq_perm": xq_perm,
            "g": g, "u": u, "a": a, "y": y, "out": out, "wq": wq, "I": I, "k": k}


def combine(y_perm, row_of, prob=None, nm: Numerics = MXFP8):
    """out[t] = sum over j = 0..k-1 of y[row_of[t][j]] (times prob[t][j] if given)."""
    y_perm = np.asarray(y_perm, dtype=np.float64)
    row_of = np.asarray(row_of)
    T, k = row_of.shape
    acc = np.zeros((T, y_perm.shape[1]))
    for j in range(k):
        term = y_perm[row_of[:, j]]
        if prob is not None:
            term = term * np.asarray(prob, dtype=np.float64)[:, j:j + 1]
        acc = acc + term
    return _bf16(acc, nm)


def swiglu_backward(dA, g, u, p):
    """Straight-through ScaledSwiGLU backward for a = silu(g) * u * p.

    Returns dg, du and dp (the row sum of dA * silu(g) * u).
    """
    s = sigmoid(g)
    sg = g * s
    dsilu = s * (1.0 + g * (1.0 - s))
    p = np.asarray(p, dtype=np.float64)[:, None]
    dg = dA * p * u * dsilu
    du = dA * p * sg
    dp = np.sum(dA * sg * u, axis=1)
    return dg, du, dp


def backward(fwd, dout, nm: Numerics = MXFP8):
    """Backward of ``forward``: dX (combined), dW_gu, dW_d, dprob.

    dY[row] = dout[src_of[row]]; per expert e:
      dA   = Q_row(dY_e) @ Q(W_d[e]^T along H)^T             (down dgrad)
      dg, du, dp from swiglu_backward with the saved bf16 g, u
      dW_d[e]  = Q_tok(dY_e)^T @ Q_tok(a_e)                   (down wgrad)
      dX_e = Q_row(dH_e) @ Q(W_gu[e]^T along 2I)^T            (gate_up dgrad)
      dW_gu[e] = Q_tok(dH_e)^T @ Q_tok(x_e)                   (gate_up wgrad)
    with dH = [dg | du]; then dx[t] = sum_j dX[row_of[t][j]], dprob[t][j] =
    dp[row_of[t][j]].
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
    dyq = q_rowwise(dy_perm, nm)
    dx_perm = np.zeros((rows, H))
    dp_perm = np.zeros(rows)
    dw_gu = np.zeros((E, 2 * I, H))
    dw_d = np.zeros((E, H, I))
    dH_all = np.zeros((rows, 2 * I))
    for e in range(E):                               # the per-expert loop
        r0, m = int(offs[e]), int(split[e])
        if m == 0:
            continue
        sl = slice(r0, r0 + m)
        dA = dyq[sl] @ wq["dT"][e].T                 # [m][I]
        dg, du, dp = swiglu_backward(dA, fwd["g"][sl], fwd["u"][sl], fwd["prob_perm"][sl])
        dH = _f32(np.concatenate([dg, du], axis=1), nm)
        dH_all[sl] = dH
        dp_perm[sl] = dp
        dw_d[e] = q_tokens(dy_perm[sl], nm).T @ q_tokens(fwd["a"][sl], nm)
        dx_perm[sl] = q_rowwise(dH, nm) @ wq["guT"][e].T
        dw_gu[e] = q_tokens(dH, nm).T @ q_tokens(fwd["x_perm"][sl], nm)
    dx_perm = _bf16(dx_perm, nm)
    dx = combine(dx_perm, perm["row_of"], nm=nm)
    dprob = _f32(dp_perm[perm["row_of"]], nm)
    return {"dx": dx, "dx_perm": dx_perm, "dw_gu": _bf16(dw_gu, nm), "dw_d": _bf16(dw_d, nm),
            "dprob": dprob, "dp_perm": dp_perm, "dH": dH_all, "dy_perm": dy_perm}

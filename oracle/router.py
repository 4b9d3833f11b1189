"""Router of the oracle on both sides (test infrastructure only).

[AutoModel], section "三板斧": each token is routed to a few of many experts;
[BioNeMo-MoE], section "MXFP8与融合MLP": the router probabilities enter the
expert FFN through ScaledSwiGLU.  The pages give no router formula; the
reading used here is the plain linear router of an MoE layer:

* logits[t][e] = sum_h x[t][h] * W_r[e][h]  (x, W_r bf16; float64 here,
  rounded to float32 -- the precision the device writes);
* the top-k selection is piecewise constant, so the gradient reaches the
  logits only through the probabilities (idx held fixed):
    renormalize:   p_j = softmax over the k selected logits
                   dl[e_j] = p_j * (dp_j - sum_i p_i dp_i), 0 elsewhere;
    plain softmax: p_j = s[e_j] with s = softmax over all E logits
                   dl[e] = s[e] * (g[e] - sum_j p_j dp_j), g[e_j] = dp_j, else 0;
* dx_router = dl @ W_r  (added to the expert FFN's dx), dW_r = dl^T @ x.
"""
from __future__ import annotations

import numpy as np

from .mxfp8 import bf16, fp32


def router_logits(x, w_r, rounded: bool = True):
    """x [T][H], w_r [E][H] -> logits [T][E]."""
    z = np.asarray(x, dtype=np.float64) @ np.asarray(w_r, dtype=np.float64).T
    return fp32(z) if rounded else z


def softmax(z):
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    ez = np.exp(z - m)
    return ez / ez.sum(axis=-1, keepdims=True)


def probs_from_logits(logits, idx, renormalize: bool = True):
    """The probabilities of the selected experts as a function of the logits (idx fixed)."""
    l64 = np.asarray(logits, dtype=np.float64)
    sel = np.take_along_axis(l64, np.asarray(idx, dtype=np.int64), axis=1)
    if renormalize:
        return softmax(sel)
    return np.take_along_axis(softmax(l64), np.asarray(idx, dtype=np.int64), axis=1)


def router_backward(logits, idx, prob, dprob, renormalize: bool = True):
    """dL/dlogits [T][E] (float64) from dL/dprob [T][k]."""
    l64 = np.asarray(logits, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    p = np.asarray(prob, dtype=np.float64)
    dp = np.asarray(dprob, dtype=np.float64)
    T, E = l64.shape
    dl = np.zeros((T, E))
    pdp = np.sum(p * dp, axis=1, keepdims=True)
    if renormalize:
        np.put_along_axis(dl, idx, p * (dp - pdp), axis=1)
    else:
        s = softmax(l64)
        g = np.zeros((T, E))
        np.put_along_axis(g, idx, dp, axis=1)
        dl = s * (g - pdp)
    return dl


def router_input_grads(dlogits, x, w_r):
    """(dx_router [T][H], dW_r [E][H]) in float64."""
    dl = np.asarray(dlogits, dtype=np.float64)
    return dl @ np.asarray(w_r, dtype=np.float64), dl.T @ np.asarray(x, dtype=np.float64)


def add_to_bf16(dx_bf16, dx_router):
    """dx of the layer: the expert FFN's bf16 dx plus the router term, rounded to bf16."""
    return bf16(np.asarray(dx_bf16, dtype=np.float64) + np.asarray(dx_router, dtype=np.float64))

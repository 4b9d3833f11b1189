"""Routing and expert-major permutation of the oracle (test infrastructure only).

[AutoModel], section "三板斧" (expert parallelism): each token is sent to a few
of many experts.  [BioNeMo-MoE], section "GroupedLinear": the grouped call
receives the tokens collected per expert together with the per-expert token
counts split_sizes; section "MXFP8与融合MLP": the router probabilities scale
the SwiGLU output.

Readings:
* Top-k by logits (exact float comparisons), ties to the lower expert index,
  slots in descending-logit order.  +0 and -0 tie.  A NaN logit ranks below
  every number (-inf included) and NaNs tie among themselves, so a row with
  fewer than k non-NaN logits still selects k distinct experts; its
  probabilities are then NaN (the pages say nothing about non-finite logits;
  this is the plainest total order that keeps the selection well defined).
* prob = softmax over the k selected logits (equivalently softmax over all E
  then renormalised over the top k).  ``renormalize=False`` keeps the plain
  softmax-over-E probabilities of the selected experts.
* Permutation: expert-major; inside one expert ascending token index (a token
  never selects the same expert twice, so this order is total).  Every expert
  segment is padded to a multiple of 128 rows; padding rows hold zeros and
  have source token -1.
"""
from __future__ import annotations

import numpy as np

ROW_PAD = 128


def route_topk(logits, k: int, renormalize: bool = True):
    """logits [T][E] float32 -> (idx int32 [T][k], prob float32 [T][k])."""
    l64 = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = l64.shape
    nan = np.isnan(l64)
    # sort keys, last one primary: NaN last, then descending logit, then ascending index
    # (np.lexsort is stable, so equal keys keep the lower index first)
    neg = np.where(nan, 0.0, -l64) + 0.0                 # + 0.0 turns -0 into +0: the two tie
    order = np.stack([np.lexsort((neg[t], nan[t])) for t in range(T)]) if T else np.zeros((0, E), np.int64)
    idx = order[:, :k]
    sel = np.take_along_axis(l64, idx, axis=1)
    m = sel[:, :1]                                       # the largest logit
    num = np.exp(sel - m)
    if renormalize:
        den = num.sum(axis=1, keepdims=True)
    else:
        den = np.exp(l64 - m).sum(axis=1, keepdims=True)
    prob = num / den
    return idx.astype(np.int32), prob.astype(np.float32)


def roundup(v, m: int = ROW_PAD):
    return ((np.asarray(v) + m - 1) // m) * m


def permute(idx, E: int):
    """Stable counting sort of the (token, slot) pairs by expert.

    Returns a dict with split_sizes int32[E], offsets_pad int32[E+1]
    (offsets_pad[e] = sum over e' < e of roundup(split_sizes[e'], 128)),
    row_of int32[T][k] (the permuted row of each pair), src_of int32[rows]
    (source token of each row, -1 on padding) and rows = offsets_pad[E].
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    split = np.bincount(idx.ravel(), minlength=E).astype(np.int64)
    offsets_pad = np.zeros(E + 1, dtype=np.int64)
    offsets_pad[1:] = np.cumsum(roundup(split))
    rows = int(offsets_pad[-1])
    key = idx * T + np.arange(T, dtype=np.int64)[:, None]  # expert-major, then token
    order = np.argsort(key.ravel(), kind="stable")
    row_of = np.empty(T * k, dtype=np.int64)
    src_of = np.full(rows, -1, dtype=np.int64)
    pos = 0
    for e in range(E):
        n = int(split[e])
        flat = order[pos:pos + n]
        r = offsets_pad[e] + np.arange(n)
        row_of[flat] = r
        src_of[r] = flat // k
        pos += n
    return {
        "split_sizes": split.astype(np.int32),
        "offsets_pad": offsets_pad.astype(np.int32),
        "row_of": row_of.reshape(T, k).astype(np.int32),
        "src_of": src_of.astype(np.int32),
        "rows": rows,
    }

"""The scaling-granularity comparison on tiny inputs: its ordering where E4M3 arithmetic fixes it.

Tokens of very different magnitude in one expert: one per-tensor scale flushes
the small tokens' activations to zero, per-token MX blocks keep them.  Without
outliers both 8-bit paths sit near E4M3's rounding error and far above the
bf16-activation path.
"""
import numpy as np

from oracle import compare_scaling as cs
from oracle import mxfp8 as mx
from oracle import routing as rt


def _inputs(seed=0, T=64, H=256, I=128, E=4):
    rng = np.random.default_rng(seed)
    x = mx.bf16(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w_gu = mx.bf16(rng.standard_normal((E, 2 * I, H)) * 0.02)
    w_d = mx.bf16(rng.standard_normal((E, H, I)) * 0.02)
    return x, logits, w_gu, w_d


def test_gaussian_inputs_both_8bit_paths_alike():
    x, logits, w_gu, w_d = _inputs()
    r = cs.compare(x, logits, w_gu, w_d, 2)
    m, p, b = (r[k]["out_rel_fro"] for k in ("mxfp8", "fp8_per_tensor", "bf16_activations"))
    assert b < m / 5 and b < p / 5
    assert 0.5 < p / m < 2.0


def test_gradients_of_small_tokens_degrade_less_than_their_outputs():
    """With the 4096x tokens, dH grows only linearly with x (dA is the same for every token),
    so the normal tokens' dH lands partly in E4M3's subnormals instead of vanishing: per-tensor
    scaling gives worse per-token dx than MX, but not the wiped-out outputs of the forward."""
    x, logits, w_gu, w_d = _inputs(1)
    dout = mx.bf16(np.random.default_rng(9).standard_normal(x.shape) * 0.01)
    r = cs.compare(cs.with_outlier_tokens(x, every=16, factor=4096.0), logits, w_gu, w_d, 2, dout)
    m, p = r["mxfp8"]["dx_token_rel_mean"], r["fp8_per_tensor"]["dx_token_rel_mean"]
    assert m < 0.15 and 1.1 * m < p < 0.5
    assert r["fp8_per_tensor"]["out_token_rel_mean"] > 0.5
    g = cs.compare(x, logits, w_gu, w_d, 2, dout)
    assert g["bf16_activations"]["dx_rel_fro"] < g["mxfp8"]["dx_rel_fro"] / 5


def test_large_tokens_wipe_out_small_ones_under_per_tensor_scaling_only():
    """Tokens 4096x the rest: a grows quadratically (silu(g)*u), so the expert's one scale
    for a flushes the normal tokens' a below E4M3's smallest subnormal; MX blocks are
    per token and keep them."""
    x, logits, w_gu, w_d = _inputs(1)
    r = cs.compare(cs.with_outlier_tokens(x, every=16, factor=4096.0), logits, w_gu, w_d, 2)
    assert r["mxfp8"]["out_token_rel_mean"] < 0.1
    assert r["fp8_per_tensor"]["out_token_rel_mean"] > 5 * r["mxfp8"]["out_token_rel_mean"]


def test_outlier_channels_stay_within_e4m3_range_for_both():
    """A 100x channel leaves the bulk of every per-tensor-scaled x in E4M3's normal range."""
    x, logits, w_gu, w_d = _inputs(1)
    r = cs.compare(cs.with_outlier_channels(x, every=128, factor=100.0), logits, w_gu, w_d, 2)
    m, p = r["mxfp8"]["out_token_rel_mean"], r["fp8_per_tensor"]["out_token_rel_mean"]
    assert m < 0.1 and p < 0.1


def test_routing_loads_are_reported():
    x, logits, w_gu, w_d = _inputs(2)
    r = cs.compare(x, logits, w_gu, w_d, 2)
    idx, _ = rt.route_topk(logits, 2)
    counts = np.bincount(idx.ravel(), minlength=4)
    assert r["loads"] == {"min": int(counts.min()), "max": int(counts.max()), "empty": int((counts == 0).sum())}

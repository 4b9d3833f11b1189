"""Test helpers: layout conversion of the device MX scales, tolerance checks.

The tile layout of MX scales is a pure index permutation (documented in
include/moe_ffn.h); converting it back to [rows][K/32] is bookkeeping, not
arithmetic of the method.
"""
import numpy as np

# float tolerance for bf16/fp32 outputs and gradients
REL_FROB = 5e-3
MAX_ABS_FRAC = 2e-2


def sf_offsets(rows: int, K: int) -> np.ndarray:
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(K // 32, dtype=np.int64)[None, :]
    return (((r >> 7) * (K >> 7) + (b >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (b & 3)


def untile_scales(flat, rows: int, K: int) -> np.ndarray:
    """Tile-layout scale bytes of a [rows][K] MX tensor -> logical [rows][K/32]."""
    flat = np.asarray(flat).reshape(-1)
    return flat[sf_offsets(rows, K)]


def tile_scales(logical) -> np.ndarray:
    logical = np.asarray(logical)
    rows, nb = logical.shape
    out = np.zeros(rows * nb, dtype=logical.dtype)
    out[sf_offsets(rows, nb * 32)] = logical
    return out


def rel_frob(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def assert_close(got, ref, name="", rel=REL_FROB, max_frac=MAX_ABS_FRAC):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rf = rel_frob(got, ref)
    mx = float(np.abs(ref).max()) if ref.size else 0.0
    ma = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert rf <= rel, f"{name}: relative Frobenius error {rf:.3e} > {rel:.1e}"
    assert ma <= max_frac * mx + 1e-30, f"{name}: max abs error {ma:.3e} > {max_frac:.0e} * {mx:.3e}"
    return rf, ma

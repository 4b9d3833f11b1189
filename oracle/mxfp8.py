"""MXFP8 codec of the oracle (test infrastructure only).

[BioNeMo-MoE], sections "MoE训练的瓶颈与TE的对应能力" and "MXFP8与融合MLP":
weights and activations are held in 8 bits and every 32 consecutive values
share one scale factor; 16-bit master values are quantized before each
low-precision GEMM.

Readings where the page is silent (each listed in the design notes):

* Element format: E4M3 -- 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
  bits; largest finite magnitude 448 (exponent 1111, mantissa 110);
  S.1111.111 is NaN; there is no infinity; subnormal step 2^-9.
* Scale: a power of two 2^e stored as the 8-bit biased exponent c = e + 127
  (code 255 = NaN).  e is the SMALLEST integer with amax <= 448 * 2^e, so no
  element of the block saturates; e is clamped to [-127, 127]; an all-zero
  block gets e = -127 (code 0).  A block holding NaN or Inf gets code 255 and
  every element the NaN code 0x7F.
* Elements: q = RNE_E4M3(x * 2^-e), round to nearest with ties to the even
  code, subnormals included, the sign of zero kept, saturating to +-448.
* The quantizer input is the float32 value available at that point (exact
  bf16 upcast for x, W and dOut; the float32 epilogue value for intermediates).

All arithmetic is exact in float64: scaling by 2^-e and the rounding grid are
powers of two.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32
E4M3_MAX = 448.0
E4M3_NAN = 0x7F
SCALE_BIAS = 127
SCALE_NAN = 255


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 code -> float64 value, from the bit-field definition."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    mf = c & 0x7
    normal = np.ldexp(1.0 + mf / 8.0, ef - 7)
    sub = np.ldexp(mf.astype(np.float64), -9)
    mag = np.where(ef == 0, sub, normal)
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def _encode_representable(v: np.ndarray) -> np.ndarray:
    """Magnitude v >= 0 that lies on the E4M3 grid -> 7-bit code."""
    m, ex = np.frexp(v)                     # v = m * 2^ex with m in [0.5, 1)
    E = ex - 1                              # floor(log2 v)
    biased = E + 7
    mant_normal = np.rint((2.0 * m - 1.0) * 8.0).astype(np.int64)
    code_normal = (biased.astype(np.int64) << 3) | mant_normal
    code_sub = np.rint(np.ldexp(v, 9)).astype(np.int64)
    code = np.where(biased >= 1, code_normal, code_sub)
    return np.where(v == 0.0, 0, code)


def e4m3_encode(y) -> np.ndarray:
    """Round float64 values to E4M3 codes: nearest, ties to even, saturating.

    The grid spacing in the binade [2^E, 2^(E+1)) is 2^(E-3) for E >= -6 and
    2^-9 below (subnormals); rounding is np.round (half to even) of y / spacing.
    """
    y = np.asarray(y, dtype=np.float64)
    neg = np.signbit(y)
    a = np.abs(y)
    nan = np.isnan(a)
    a_fin = np.where(nan, 0.0, np.minimum(a, 2.0 * E4M3_MAX))  # Inf saturates below
    _, ex = np.frexp(a_fin)
    E = ex - 1
    step_exp = np.maximum(E, -6) - 3
    q = np.round(np.ldexp(a_fin, -step_exp))
    v = np.minimum(np.ldexp(q, step_exp), E4M3_MAX)
    code = _encode_representable(v) | (neg.astype(np.int64) << 7)
    code = np.where(nan, E4M3_NAN | (neg.astype(np.int64) << 7), code)
    return code.astype(np.uint8)


def scale_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127].

    amax = 0 gives -127.  Non-finite amax is returned as +128 (a marker; the
    caller turns it into the NaN scale code).
    """
    amax = np.asarray(amax, dtype=np.float64)
    bad = ~np.isfinite(amax)
    a = np.where(bad | (amax == 0.0), 1.0, amax)
    _, ex = np.frexp(a)
    e = (ex - 1) - 8                        # 448 = 1.75 * 2^8
    e = np.where(a > np.ldexp(E4M3_MAX, e), e + 1, e)
    e = np.clip(e, -127, 127)
    e = np.where(amax == 0.0, -127, e)
    return np.where(bad, 128, e).astype(np.int64)


def quantize_blocks(x, axis: int = -1):
    """MX-quantize along ``axis`` in blocks of 32 consecutive values.

    Returns (codes uint8 with x's shape, scale codes uint8 with the axis
    length divided by 32).  The axis length must be a multiple of 32; callers
    pad partial blocks with zeros (zeros never change a block's amax).
    """
    x = np.asarray(x, dtype=np.float64)
    xm = np.moveaxis(x, axis, -1)
    n = xm.shape[-1]
    if n % BLOCK:
        raise ValueError("axis length must be a multiple of 32")
    xb = xm.reshape(xm.shape[:-1] + (n // BLOCK, BLOCK))
    amax = np.max(np.abs(xb), axis=-1)      # NaN propagates
    e = scale_exponent(amax)
    bad = e == 128
    e_use = np.where(bad, 0, e)
    y = np.ldexp(xb, -e_use[..., None])
    codes = e4m3_encode(y)
    codes = np.where(bad[..., None], np.uint8(E4M3_NAN), codes)
    sc = np.where(bad, SCALE_NAN, e_use + SCALE_BIAS).astype(np.uint8)
    codes = np.moveaxis(codes.reshape(xm.shape), -1, axis)
    sc = np.moveaxis(sc, -1, axis)
    return codes, sc


def dequantize_blocks(codes, scales, axis: int = -1) -> np.ndarray:
    """Inverse map: decode(code) * 2^(scale - 127), scale code 255 -> NaN."""
    v = e4m3_decode(codes)
    s = np.asarray(scales).astype(np.int64)
    f = np.where(s == SCALE_NAN, np.nan, np.ldexp(1.0, np.where(s == SCALE_NAN, 0, s - SCALE_BIAS)))
    f = np.repeat(f, BLOCK, axis=axis)
    return v * f


def fp32(x) -> np.ndarray:
    """Round to the nearest float32 (the precision a quantizer receives)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16(x) -> np.ndarray:
    """Round float64 -> float32 -> bfloat16 (both RNE), returned as float64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    rnd = ((u >> 16) & 1) + 0x7FFF
    u2 = ((u + rnd) >> 16) << 16
    out = u2.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(nan, np.nan, out)

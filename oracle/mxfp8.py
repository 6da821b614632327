"""MXFP8 block quantisation, float64 reference (test infrastructure only).

Format.  The pages name the mode only ("MXFP8", weights pre-quantised with
``ops.mxfp8_quantize``: *Mixture-of-Kittens (MoK)*, "Core concepts" table,
MXFP8 row).  The element and scale types and the block size are the OCP
Microscaling (MX) v1.0 MXFP8 format: E4M3 elements (the "FN" variant: bias 7,
no infinities, largest finite 448) sharing one E8M0 scale (a biased power of
two, bias 127) per block of 32 consecutive elements along the GEMM's K axis.

Scale rule (the OCP MX conversion): shared exponent
``X = floor(log2(amax)) - 8`` (8 is the largest normal exponent of E4M3),
clamped to the E8M0 range [-127, 127]; an all-zero block takes X = -127.
Elements are ``RNE(v / 2^X)`` on the E4M3 grid, saturating at +-448.

Encoding of zero: a negative input that rounds to zero keeps its sign bit
(code 0x80); positive zero is code 0x00.
"""

from __future__ import annotations

import numpy as np

BLOCK = 32
E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6
E4M3_MANT_BITS = 3
E8M0_BIAS = 127
E4M3_EMAX = 8  # exponent of the largest normal E4M3 value, 448 = 1.75 * 2^8


def e4m3_decode(codes):
    """Value of each E4M3 code (0..255) from its bit fields; NaN for 0x7F/0xFF."""
    codes = np.asarray(codes, dtype=np.int64)
    sign = np.where((codes >> 7) & 1, -1.0, 1.0)
    exp = (codes >> 3) & 0xF
    man = (codes & 0x7).astype(np.float64)
    val = np.where(exp == 0,
                   man / 8.0 * 2.0 ** E4M3_MIN_NORMAL_EXP,
                   (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0))
    val = np.where((exp == 15) & ((codes & 7) == 7), np.nan, val)
    return sign * val


def e4m3_round(v):
    """Round float64 values to the nearest E4M3 value, ties to even, saturating.

    Written from the format's definition: in the binade [2^e, 2^(e+1)) (e no
    lower than the subnormal floor -6) the spacing is 2^(e-3); ``np.round``
    rounds halves to even, which is the even-mantissa rule because the
    quotient is the integer significand.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        _, ex = np.frexp(a)           # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)
    quantum = np.exp2((e - E4M3_MANT_BITS).astype(np.float64))
    q = np.round(a / quantum) * quantum
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_encode(v):
    """Code (0..255) of values that are already on the E4M3 grid."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = np.signbit(v).astype(np.int64) << 7
    with np.errstate(divide="ignore"):
        _, ex = np.frexp(a)
    e = ex - 1
    normal = a >= 2.0 ** E4M3_MIN_NORMAL_EXP
    # normal: a = (1 + m/8) 2^e, field = e + 7
    m_norm = np.where(normal, np.round((a / np.exp2(e.astype(np.float64)) - 1.0) * 8.0), 0)
    f_norm = np.where(normal, e + 7, 0)
    # subnormal: a = m/8 * 2^-6
    m_sub = np.round(a / 2.0 ** E4M3_MIN_NORMAL_EXP * 8.0)
    mant = np.where(normal, m_norm, m_sub).astype(np.int64)
    field = np.where(normal, f_norm, 0).astype(np.int64)
    return (sign | (field << 3) | mant).astype(np.uint8)


def scale_exponent(amax):
    """Shared block exponent X of the OCP MX rule (int64 array)."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        _, ex = np.frexp(amax)
    x = (ex - 1) - E4M3_EMAX
    x = np.clip(x, -E8M0_BIAS, E8M0_BIAS)
    return np.where(amax == 0.0, -E8M0_BIAS, x).astype(np.int64)


def quantize(a, axis):
    """Quantise ``a`` in blocks of 32 along ``axis``.

    Returns ``(codes, scale_codes, dequantised)``: codes has ``a``'s shape
    (uint8), scale_codes has ``a``'s shape with ``axis`` divided by 32
    (uint8, E8M0 = X + 127), dequantised = decoded element * 2^X (float64).
    The length along ``axis`` must be a multiple of 32.
    """
    a = np.asarray(a, dtype=np.float64)
    a_m = np.moveaxis(a, axis, -1)
    K = a_m.shape[-1]
    if K % BLOCK:
        raise ValueError(f"length {K} along axis {axis} is not a multiple of {BLOCK}")
    blocks = a_m.reshape(a_m.shape[:-1] + (K // BLOCK, BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    X = scale_exponent(amax)
    scale = np.exp2(X.astype(np.float64))[..., None]
    q = e4m3_round(blocks / scale)
    deq = (q * scale).reshape(a_m.shape)
    codes = e4m3_encode(q).reshape(a_m.shape)
    return (np.moveaxis(codes, -1, axis),
            np.moveaxis((X + E8M0_BIAS).astype(np.uint8), -1, axis),
            np.moveaxis(deq, -1, axis))


def qdq(a, axis):
    """Quantise then dequantise along ``axis`` (float64 result)."""
    return quantize(a, axis)[2]


def qdq_rows_padded(a, axis=0):
    """Quantise along ``axis`` after zero-padding it to a multiple of 32.

    Used for the weight-gradient operands, whose K axis is an expert's routed
    rows; padding rows are zero and do not change any block's amax.
    """
    a = np.asarray(a, dtype=np.float64)
    n = a.shape[axis]
    pad = (-n) % BLOCK
    if pad:
        widths = [(0, 0)] * a.ndim
        widths[axis] = (0, pad)
        a = np.pad(a, widths)
    d = qdq(a, axis)
    return np.take(d, np.arange(n), axis=axis)

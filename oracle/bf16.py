"""Exact rounding of real (fp64) values to bfloat16 (oracle side).

bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the fp32
exponent range.  The V-Smooth block mean is "kept as a 16-bit mean"
(VC-Attention news article, section 2 "V-Smooth", third step); the reading
taken is bfloat16, rounded once, to nearest-even, from the exact real mean.
Attention outputs are bf16 as well (TeleFuser FP8 Sol-Attn blog, boundary
table: attention returns BF16).
"""
from __future__ import annotations

import numpy as np

_BF16_MIN_NORMAL_EXP = -126


def round_to_bf16(d) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value, ties to even.

    Returns the rounded values as fp64.  The rounding is done directly from
    fp64 (a single rounding): in the binade 2^e <= |d| < 2^(e+1) the grid
    spacing is 2^(e-7); below the normal range it is the subnormal spacing
    2^-133.  Values beyond the bf16 range become +-inf (never reached by the
    data this oracle sees).
    """
    d = np.asarray(d, dtype=np.float64)
    a = np.abs(d)
    _, k = np.frexp(a)
    e = np.maximum(k - 1, _BF16_MIN_NORMAL_EXP)
    q = np.ldexp(1.0, e - 7)
    r = np.rint(a / q) * q
    r = np.where(r > 3.3895313892515355e38, np.inf, r)
    return np.copysign(r, d)


def bf16_bits(values) -> np.ndarray:
    """uint16 bit patterns of values that are already exactly bf16."""
    f = np.asarray(values, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    """fp64 values of uint16 bf16 bit patterns (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)

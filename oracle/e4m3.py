"""Bit-level OCP E4M3FN codec (oracle side; test infrastructure only).

Format facts used (P-Cast Precision review, section 3 "FP8 E4M3 precision
bottleneck"; TeleFuser FP8 Sol-Attn blog, section "FP8 Preparation for
attention", where scales divide by 448):
  * 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, so every normal
    binade holds 8 evenly spaced values (12.5 % relative step);
  * largest finite magnitude 448 = 1.75 * 2^8 (code 0x7E); code 0x7F and
    0xFF are NaN, there is no infinity (the "FN" variant);
  * subnormals are k * 2^-9 for k = 1..7, so the smallest positive value is
    2^-9 and anything below 2^-10 rounds to zero (the review's underflow
    condition p*S < 2^-10).

Encoding rounds to nearest, ties to even, and saturates finite overflow to
+-448 ("satfinite").  A negative value that rounds to zero keeps its sign
(code 0x80).  These are the semantics of the E4M3 conversion the review and
the TeleFuser prep use; the choice of saturation over NaN on overflow is the
reading taken here (the pages never overflow: every scale maps the block
maximum to exactly 448).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9
NAN_CODE = 0x7F


def decode_table() -> np.ndarray:
    """Exact value of every one of the 256 codes, as fp64 (NaN for 0x7F/0xFF).

    Built from the field layout alone: value = (-1)^s * 2^(e-7) * (1 + m/8)
    for e >= 1, and (-1)^s * 2^-6 * (m/8) for e == 0.
    """
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = (code >> 7) & 1
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            v = np.nan
        elif e == 0:
            v = (m / 8.0) * 2.0 ** -6
        else:
            v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
        out[code] = -v if s else v
    return out


_TABLE = decode_table()


def decode(codes) -> np.ndarray:
    """Exact fp64 value of E4M3 codes (any integer array of bytes)."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x) -> np.ndarray:
    """E4M3 code (uint8) of each value of ``x``, round-to-nearest-even, satfinite.

    ``x`` holds fp32 values (the kernels convert fp32 registers); they are
    carried exactly in fp64 here.  Steps:
      1. a = |x|; the binade exponent e satisfies 2^e <= a < 2^(e+1);
         below the normal range the subnormal quantum 2^-9 is used, which is
         also the quantum of the lowest normal binade (e = -6).
      2. the grid spacing in that binade is q = 2^(e-3) (3 mantissa bits);
         r = rint(a / q) * q rounds to the nearest grid point, ties to even
         (numpy's rint is round-half-even; a / q is exact).
      3. r > 448 saturates to 448.
      4. the code is (e_r + 7) << 3 | mantissa for normal r, and r * 2^9 for
         subnormal r (which yields 8 = code of 2^-6 when a subnormal rounds
         up into the normal range, consistent with the field layout).
    NaN maps to 0x7F; +-inf saturates to +-448.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    a = np.where(np.isinf(a), E4M3_MAX, a)
    _, k = np.frexp(a)                      # a = f * 2^k, f in [0.5, 1)
    e = np.maximum(k - 1, -6)
    q = np.ldexp(1.0, e - 3)
    r = np.rint(a / q) * q
    r = np.minimum(r, E4M3_MAX)
    _, k2 = np.frexp(r)
    e2 = k2 - 1
    normal = r >= E4M3_MIN_NORMAL
    mant = np.where(normal, (r / np.ldexp(1.0, e2) - 1.0) * 8.0, 0.0)
    code_normal = ((e2 + 7) << 3) + mant.astype(np.int64)
    code_sub = (r * 2.0 ** 9).astype(np.int64)
    code = np.where(normal, code_normal, code_sub).astype(np.int64)
    code = np.where(sign, code | 0x80, code)
    code = np.where(nan, NAN_CODE, code)
    return code.astype(np.uint8)


def quantum_at(v: float) -> float:
    """Spacing of the E4M3 grid in the binade holding positive value ``v``."""
    if v < E4M3_MIN_NORMAL:
        return E4M3_MIN_SUBNORMAL
    _, k = np.frexp(v)
    return 2.0 ** (int(k) - 1 - 3)

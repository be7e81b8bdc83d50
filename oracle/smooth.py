"""Sequence-mean smoothing of K and V (test infrastructure only).

Follows the TeleFuser FP8 Sol-Attn blog, section "Diffusion precision guards"
(attention sequence-mean smoothing): for every attention head the prep takes
K' = K - mean_T(K) and V' = V - mean_T(V), with fp32 statistics, fused into the
E4M3 preparation.  Shifting K adds the same constant to every logit of a query
row, so the softmax is unchanged; the softmax weights of a row sum to one, so
adding mean_T(V) back to the attention output restores it.  The residual mean
bias of V measured after the E4M3 rounding is compensated as well.

Readings where the page is silent:
  * mean_T is the exact mean of one (batch, head, channel) over the T tokens,
    rounded once to fp32 (nearest even): it does not depend on a summation
    order;
  * K' = fl32(K - kbar) and V' = fl32(V - vbar): one fp32 subtraction, the
    centred values then go through the usual block quantisation;
  * the V bias of a channel is b_c = mean_t(Vhat'[t,c] - V'[t,c]), Vhat' the
    dequantised V' (residual code times the channel scale, plus the block mean
    with V-Smooth); the output row gets + vbar_c - b_c, added in fp32 before
    the output is rounded to bf16;
  * modes: smooth = 0 (none), 1 (K), 2 (K and V); the bias correction is
    independent of the mode.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

from .e4m3 import decode

SMOOTH_NONE, SMOOTH_K, SMOOTH_KV = 0, 1, 2


def round_fraction_to_f32(q: Fraction) -> np.float32:
    """Nearest fp32 value to a rational, ties to even (normal range)."""
    if q == 0:
        return np.float32(0.0)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (e - 23)
    n = round(a / quantum)          # Fraction.__round__: half to even
    v = np.float32(float(n * quantum))
    return np.float32(-v) if q < 0 else v


def seq_mean_f32(x: np.ndarray) -> np.ndarray:
    """Exact per-channel mean over the rows of x [T, C], rounded once to fp32.

    x holds fp64 values that are exact (bf16 inputs).  The column sum is taken
    in fp64 when that is exact (8-bit significands, at most 2^17 rows: a span
    of at most 53 - 8 - 17 = 28 binades), else as an exact rational sum.
    """
    x = np.asarray(x, dtype=np.float64)
    T, C = x.shape
    out = np.zeros(C, dtype=np.float32)
    _, k = np.frexp(x)
    nz = x != 0
    kmax = np.where(nz, k, -10**6).max(axis=0)
    kmin = np.where(nz, k, 10**6).min(axis=0)
    fast = ((kmax - kmin) <= 53 - 8 - max(1, math.ceil(math.log2(max(T, 2))))) | (~nz.any(axis=0))
    sums = x.sum(axis=0)
    for c in range(C):
        s = Fraction(float(sums[c])) if fast[c] else sum(Fraction(float(v)) for v in x[:, c])
        out[c] = round_fraction_to_f32(s / T)
    return out


def center(x: np.ndarray, mean_f32: np.ndarray) -> np.ndarray:
    """fl32(x - mean): the centred rows, as fp64 arrays of fp32 values."""
    return (np.asarray(x, dtype=np.float32) - np.asarray(mean_f32, dtype=np.float32)[None, :]) \
        .astype(np.float32).astype(np.float64)


def v_bias(vq: np.ndarray, sv: np.ndarray, mean_blk: np.ndarray, vprime: np.ndarray) -> np.ndarray:
    """Per-channel mean of (dequantised V' - V') over the T valid rows, exact (fp64 [128]).

    vq [128, Tpad] residual codes in permuted order, sv [128] channel scales,
    mean_blk [nV, 128] block means (zeros without V-Smooth), vprime [T, 128]
    the centred rows in the same (permuted) order.
    """
    T = vprime.shape[0]
    deq = decode(vq[:, :T]).T * np.asarray(sv, dtype=np.float64)[None, :] \
        + np.repeat(np.asarray(mean_blk, dtype=np.float64), 128, axis=0)[:T]
    return (deq - vprime).mean(axis=0)

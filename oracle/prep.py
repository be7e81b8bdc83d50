"""Stage 1 oracle: FP8 preparation of post-RoPE bf16 Q, K, V (test infrastructure only).

Follows
  * TeleFuser FP8 Sol-Attn blog, section "FP8 Preparation for attention":
    one scale per (batch, head, 64-token block) for Q and K,
    s = max|block| / 448; V scale per (batch, head, channel) over all tokens;
    V stored token-contiguous for the K-major PV product.
  * FPSAttention article, section 2.1: the FP8 quantiser multiplies by the
    group scale before the FP8 conversion (X * s_g), so the kernel-side
    reading is "multiply by 448 / amax", computed once per group.
  * VC-Attention news article, section 2 "V-Smooth": V rows are gathered by a
    token permutation, each 128-row block's mean mu_j = (1/B_v) V'_j^T 1 is
    subtracted and only the residual R_j = V'_j - 1 mu_j^T is quantised; the
    mean is kept as a 16-bit vector per block.

Readings taken where the pages are silent:
  * scale arithmetic is IEEE fp32 with round-to-nearest, no fused multiply-add:
    s = fl32(a / 448), inv = fl32(448 / a), code = E4M3(fl32(x * inv));
  * a block (or a channel) whose maximum is 0 gets s = 0 and inv = 0, so its
    codes encode +-0;
  * the token permutation reorders K and V rows together (attention is only
    preserved if keys and values move as pairs); Q and the output keep the
    original order;
  * the 16-bit mean is bfloat16, the exact real mean rounded once to nearest
    even; a ragged last block averages over its valid rows only;
  * the residual R = fl32(V' - mu) is quantised with one scale per
    (batch, head, channel) over all tokens, the granularity the TeleFuser V
    scale uses and the one that lets the channel scale be applied after all
    PV products; with V-Smooth off, mu = 0 and R = V'.

Arrays: bf16 tensors are passed as uint16 bit patterns, shape [B, T, H, 128].
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

from .bf16 import bf16_bits, bf16_from_bits, round_to_bf16
from .e4m3 import E4M3_MAX, encode

QK_BLOCK = 64     # tokens per Q/K scale block
V_BLOCK = 128     # rows per V-Smooth block (B_v)
HEAD_DIM = 128

_F448 = np.float32(E4M3_MAX)


def _scale_pair(a: np.float32):
    """(s, inv) for a block maximum a, in fp32: s = a/448, inv = 448/a (0 when a == 0)."""
    a = np.float32(a)
    if a == 0:
        return np.float32(0.0), np.float32(0.0)
    return np.float32(a / _F448), np.float32(_F448 / a)


def quantize_qk_head(x: np.ndarray):
    """Block-quantise one (batch, head) slice of Q or K.

    x: fp32/fp64 array [T, 128] of bf16 values, rows in stored order.
    Returns (codes uint8 [T, 128], scales fp32 [ceil(T/64)]).
    """
    x = np.asarray(x, dtype=np.float32)
    T = x.shape[0]
    nb = -(-T // QK_BLOCK)
    codes = np.zeros((T, HEAD_DIM), dtype=np.uint8)
    scales = np.zeros(nb, dtype=np.float32)
    for j in range(nb):
        blk = x[j * QK_BLOCK:(j + 1) * QK_BLOCK]
        a = np.max(np.abs(blk))
        s, inv = _scale_pair(a)
        scales[j] = s
        y = (blk * inv).astype(np.float32)          # fp32 product, round to nearest
        codes[j * QK_BLOCK:(j + 1) * QK_BLOCK] = encode(y)
    return codes, scales


def prep_qk(x_bits: np.ndarray, perm: np.ndarray | None = None, heads=None):
    """Quantise a whole Q or K tensor.

    x_bits: uint16 [B, T, H, 128] bf16 bit patterns.
    perm:   int [B, H, T] token permutation applied to the rows of each
            (batch, head) before blocking (used for K), or None.
    heads:  optional iterable of (b, h) pairs to compute; others stay zero.
    Returns (codes uint8 [B, T, H, 128], scales fp32 [B, H, ceil(T/64)]).
    """
    B, T, H, D = x_bits.shape
    assert D == HEAD_DIM
    nb = -(-T // QK_BLOCK)
    codes = np.zeros((B, T, H, D), dtype=np.uint8)
    scales = np.zeros((B, H, nb), dtype=np.float32)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        x = bf16_from_bits(x_bits[b, :, h, :])
        if perm is not None:
            x = x[np.asarray(perm[b, h], dtype=np.int64)]
        c, s = quantize_qk_head(x)
        codes[b, :, h, :] = c
        scales[b, h] = s
    return codes, scales


def _round_fraction_to_bf16(q: Fraction) -> float:
    """Exact round-to-nearest-even of a rational to bfloat16: grid spacing
    2^(e-7) in the binade [2^e, 2^(e+1)), the subnormal spacing 2^-133 below
    2^-126 (a bf16 block mean is a bf16 value at every magnitude)."""
    if q == 0:
        return 0.0
    a = abs(q)
    e = math.floor(math.log2(a.numerator)) - math.floor(math.log2(a.denominator))
    # fix e so that 2^e <= a < 2^(e+1)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 7)
    n = round(a / quantum)          # Fraction.__round__ rounds half to even
    v = float(n * quantum)
    return -v if q < 0 else v


def _fp64_sum_is_exact(blocks: np.ndarray) -> np.ndarray:
    """Per (block, channel): is the fp64 sum of this column exact?

    blocks: [nblk, rows, 128].  The values are bf16 (8-bit significands) or,
    after sequence-mean centring, fp32 (24-bit); with at most 128 terms an
    fp64 sum is exact when the binary exponents of the nonzero terms span at
    most 53 - 7 - 24 = 22 (fp32) or 38 (bf16) binades.
    """
    _, k = np.frexp(blocks)
    nz = blocks != 0
    kmax = np.where(nz, k, -10**6).max(axis=1)
    kmin = np.where(nz, k, 10**6).min(axis=1)
    is_bf16 = np.all(blocks.astype(np.float32).view(np.uint32) & 0xFFFF == 0, axis=1)
    return (kmax - kmin <= np.where(is_bf16, 38, 22)) | (~nz.any(axis=1))


def block_means(vp: np.ndarray) -> np.ndarray:
    """bf16 V-Smooth block means of permuted rows vp [T, 128] (fp64 values).

    mu_j = bf16_RNE( exact sum of the valid rows of block j / their count ).
    Full blocks have 128 rows, so sum / 128 is exact in fp64 and rounds once;
    a ragged last block is divided and rounded in exact rational arithmetic.
    Returns fp64 [ceil(T/128), 128] holding bf16 values.
    """
    T = vp.shape[0]
    nV = -(-T // V_BLOCK)
    mu = np.zeros((nV, HEAD_DIM), dtype=np.float64)
    full = T // V_BLOCK
    if full:
        blocks = vp[:full * V_BLOCK].reshape(full, V_BLOCK, HEAD_DIM)
        sums = blocks.sum(axis=1)
        exact = _fp64_sum_is_exact(blocks)
        mu[:full] = round_to_bf16(sums / V_BLOCK)
        for j, c in zip(*np.nonzero(~exact)):
            s = sum(Fraction(float(x)) for x in blocks[j, :, c])
            mu[j, c] = _round_fraction_to_bf16(s / V_BLOCK)
    if full < nV:
        tail = vp[full * V_BLOCK:]
        cnt = tail.shape[0]
        exact = _fp64_sum_is_exact(tail[None])[0]
        for c in range(HEAD_DIM):
            col = tail[:, c]
            s = Fraction(float(np.sum(col))) if exact[c] else sum(Fraction(float(x)) for x in col)
            mu[full, c] = _round_fraction_to_bf16(s / cnt)
    return mu


def prep_v_head(v: np.ndarray, perm_h: np.ndarray | None, vsmooth: bool, vbar=None):
    """V-Smooth preparation of one (batch, head) slice.

    v: fp64 [T, 128] bf16 values in original token order.
    vbar: optional fp32 [128] sequence mean; the rows are centred first,
    V' = fl32(V - vbar) (sequence-mean smoothing, oracle/smooth.py).
    Returns dict with
      mean  fp64 [nV, 128] (bf16 values; zeros when vsmooth is off)
      vq    uint8 [128, Tpad] residual codes, token-contiguous, pads = 0
      sv    fp32 [128] per-channel residual scale amax/448
      amax  fp32 [128]
      resid fp32 [T, 128] residual R (for diagnostics)
    """
    T = v.shape[0]
    nV = -(-T // V_BLOCK)
    if vbar is not None:
        v = (np.asarray(v, dtype=np.float32) - np.asarray(vbar, dtype=np.float32)[None, :]) \
            .astype(np.float32).astype(np.float64)
    vp = v[np.asarray(perm_h, dtype=np.int64)] if perm_h is not None else v
    mu = block_means(vp) if vsmooth else np.zeros((nV, HEAD_DIM))
    mu_rows = np.repeat(mu, V_BLOCK, axis=0)[:T]
    resid = (vp.astype(np.float32) - mu_rows.astype(np.float32)).astype(np.float32)
    amax = np.max(np.abs(resid), axis=0).astype(np.float32)
    sv = np.zeros(HEAD_DIM, dtype=np.float32)
    inv = np.zeros(HEAD_DIM, dtype=np.float32)
    for c in range(HEAD_DIM):
        sv[c], inv[c] = _scale_pair(amax[c])
    codes = encode((resid * inv[None, :]).astype(np.float32))
    vq = np.zeros((HEAD_DIM, nV * V_BLOCK), dtype=np.uint8)
    vq[:, :T] = codes.T
    return dict(mean=mu, vq=vq, sv=sv, amax=amax, resid=resid, vprime=vp)


def prep_v(v_bits: np.ndarray, perm: np.ndarray | None, vsmooth: bool, heads=None):
    """V preparation for a whole tensor (or a subset of (b, h) pairs).

    Returns (mean_bits uint16 [B,H,nV,128], vq uint8 [B,H,128,Tpad],
             sv fp32 [B,H,128], amax fp32 [B,H,128]).
    """
    B, T, H, D = v_bits.shape
    nV = -(-T // V_BLOCK)
    mean_bits = np.zeros((B, H, nV, D), dtype=np.uint16)
    vq = np.zeros((B, H, D, nV * V_BLOCK), dtype=np.uint8)
    sv = np.zeros((B, H, D), dtype=np.float32)
    amax = np.zeros((B, H, D), dtype=np.float32)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        v = bf16_from_bits(v_bits[b, :, h, :])
        r = prep_v_head(v, None if perm is None else perm[b, h], vsmooth)
        mean_bits[b, h] = bf16_bits(r["mean"])
        vq[b, h] = r["vq"]
        sv[b, h] = r["sv"]
        amax[b, h] = r["amax"]
    return mean_bits, vq, sv, amax

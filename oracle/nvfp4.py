"""4-bit (NVFP4) PV product: E2M1 elements with a scale per 16 elements
(test infrastructure only).

Follows the VC-Attention news article, section 3 (last paragraph) and the
Figure 6 discussion: on workstation Blackwell the method runs a 4-bit
configuration that uses V-Smooth but not the direct probability cast,
because 4-bit floating-point probabilities need a scale for every 16
elements; section 2 notes that removing the block mean lets the same 4- or
8-bit grid resolve the residual more finely.  The abstract page lists the
workstation cards among the targets.

Readings (the pages give no 4-bit formulas):
  * element format E2M1 (0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives), round to
    nearest with ties to the even code, saturating at 6; a negative value
    that rounds to 0 keeps its sign (code 8), as E4M3 does;
  * one scale per 16 elements in unsigned E4M3 (UE4M3), round to nearest
    even, saturating at 448 (the NVFP4 layout);
  * two-level scaling of the V residual (after the V-Smooth block mean):
    channel c gets s_c = fl32(amax_c / 2688) and G_c = fl32(2688 / amax_c)
    (2688 = 6 x 448); a block b of 16 tokens gets sf = UE4M3(fl32(fl32(a_b *
    G_c) * fl32(1/6))) with a_b its largest |R|, and every element the code
    E2M1(fl32(R * fl32(G_c / sf))); the decoded residual is e2m1 * sf * s_c;
  * P: p = fl32(2688 * exp(x - m)) (a static P scale of 6 x 448 keeps the block
    scales in the normal UE4M3 range), a block of 16 keys of the 128-key tile
    gets sf = UE4M3(fl32(a_b * fl32(1/6))) and every element E2M1(fl32(p *
    fl32(1/sf))); the decoded P is e2m1 * sf and the row sum is the sum of the
    decoded values (keys past T are absent from their block);
  * Q and K stay E4M3 (the 8-bit preparation): the pages do not state the QK
    precision of the 4-bit configuration.
"""
from __future__ import annotations

import numpy as np

from . import e4m3
from . import prep as OP

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_MIDPOINTS = (E2M1_VALUES[:-1] + E2M1_VALUES[1:]) / 2          # 0.25 0.75 1.25 1.75 2.5 3.5 5
FP4_PSCALE = 2688.0                                              # 6 x 448
BLOCK = 16
SIXTH = np.float32(1.0) / np.float32(6.0)                        # fl32(1/6)


def e2m1_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    v = E2M1_VALUES[c & 7]
    return np.where(c & 8, -v, v)


def e2m1_encode(x) -> np.ndarray:
    """Nearest E2M1 code (ties to the even code, |x| >= 6 -> 6), sign kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    code = np.zeros(a.shape, dtype=np.int64)
    for j, mid in enumerate(_MIDPOINTS):
        code += (a > mid)
        if j % 2 == 1:                  # a tie between codes j (odd) and j+1 (even) goes up
            code += (a == mid)
    return (code | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def ue4m3_encode(x) -> np.ndarray:
    """UE4M3 scale code of non-negative fp32 values (E4M3 rounding, satfinite)."""
    return e4m3.encode(np.asarray(x, dtype=np.float32))


def _blocks(x: np.ndarray, valid: int) -> list:
    return [(s, min(s + BLOCK, valid)) for s in range(0, valid, BLOCK)]


def quantize_residual(resid: np.ndarray):
    """NVFP4 V residual of one head: resid fp32 [T, 128] -> (codes uint8 [128, Tpad],
    sf codes uint8 [128, Tpad // 16], s_c fp32 [128], amax fp32 [128])."""
    T = resid.shape[0]
    nV = -(-T // OP.V_BLOCK)
    Tpad = nV * OP.V_BLOCK
    amax = np.max(np.abs(resid), axis=0).astype(np.float32) if T else np.zeros(OP.HEAD_DIM, np.float32)
    codes = np.zeros((OP.HEAD_DIM, Tpad), dtype=np.uint8)
    sfc = np.zeros((OP.HEAD_DIM, Tpad // BLOCK), dtype=np.uint8)
    s_c = np.zeros(OP.HEAD_DIM, dtype=np.float32)
    for c in range(OP.HEAD_DIM):
        if amax[c] == 0:
            continue
        s_c[c] = np.float32(amax[c] / np.float32(FP4_PSCALE))
        G = np.float32(np.float32(FP4_PSCALE) / amax[c])
        col = resid[:, c].astype(np.float32)
        for s, e in _blocks(col, T):
            a = np.float32(np.max(np.abs(col[s:e])))
            sf = ue4m3_encode(np.float32(np.float32(a * G) * SIXTH))
            sfc[c, s // BLOCK] = sf
            sfv = np.float32(e4m3.decode(sf))
            if sfv == 0:
                continue
            r = np.float32(G / sfv)
            codes[c, s:e] = e2m1_encode((col[s:e] * r).astype(np.float32))
    return codes, sfc, s_c, amax


def prep_v_head_fp4(v: np.ndarray, perm_h, vsmooth: bool, vbar=None):
    """V-Smooth preparation with an NVFP4 residual (same gather, block means and
    residual as the 8-bit preparation, oracle/prep.py)."""
    base = OP.prep_v_head(v, perm_h, vsmooth, vbar=vbar)
    codes, sfc, s_c, amax = quantize_residual(base["resid"])
    return dict(mean=base["mean"], v4=codes, sf=sfc, sc=s_c, amax=amax, resid=base["resid"],
                vprime=base["vprime"])


def vhat_fp4(v4: np.ndarray, sfc: np.ndarray, s_c: np.ndarray, mean: np.ndarray, T: int) -> np.ndarray:
    """Decoded V [T, 128] (fp64): e2m1 * block scale * channel scale + block mean."""
    sfv = e4m3.decode(sfc)                                           # [128, Tpad/16]
    r = e2m1_decode(v4[:, :T]) * np.repeat(sfv, BLOCK, axis=1)[:, :T] * s_c[:, None].astype(np.float64)
    mu = np.repeat(mean, OP.V_BLOCK, axis=0)[:T]
    return r.T + mu


def pcast_fp4(x_minus_m: np.ndarray) -> np.ndarray:
    """Decoded 4-bit P of one tile: x_minus_m fp64 [R, n] (n <= 128 keys of the tile,
    natural-log units) -> P^ fp64 [R, n], blocks of 16 keys from the tile start."""
    p = (FP4_PSCALE * np.exp(x_minus_m)).astype(np.float32)
    out = np.zeros(p.shape)
    for s, e in _blocks(p[0] if p.ndim > 1 else p, p.shape[-1]):
        a = np.max(p[:, s:e], axis=1).astype(np.float32)
        sf = ue4m3_encode((a * SIXTH).astype(np.float32))
        sfv = e4m3.decode(sf).astype(np.float32)
        with np.errstate(divide="ignore"):
            r = np.where(sfv > 0, (np.float32(1.0) / np.where(sfv > 0, sfv, 1)).astype(np.float32), 0)
        q = e2m1_encode((p[:, s:e] * r[:, None].astype(np.float32)).astype(np.float32))
        out[:, s:e] = e2m1_decode(q) * sfv[:, None].astype(np.float64)
    return out

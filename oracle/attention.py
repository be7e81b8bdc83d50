"""Stage 2 oracle: emulated FP8 attention, exact attention, P-only emulation.

Test infrastructure only.

What the emulation follows
  * TeleFuser FP8 Sol-Attn blog, section "SM90 CuTe mainloop": QK on E4M3
    operands, the block scales applied to the fp32 scores before the online
    softmax; P converted to E4M3 and multiplied with token-contiguous E4M3 V;
    the V channel scale applied to the output accumulator after all PV
    products; one shared online-softmax state (row max, row sum, output
    accumulator); output in bf16.
  * VC-Attention news article, section 2 "V-Smooth" (third step): the block
    mean is restored as the rank-one term r_ij mu_j^T, where r_ij is the row
    sum of the block's probabilities that the online softmax already keeps,
    sharing the accumulator's rescaling.  sum_t P_t (R_t s_v + mu_blk(t)) is
    the same sum written per key, which is how it is computed here.
  * VC-Attention news article, section 3 "ExpCast": the E4M3 probability
    code is c = round(8 z + 56 + beta), z the base-2 log of the probability,
    beta = -0.35, replacing the exponential and the format conversion.
  * FPSAttention article, section 3.1: P is cast with a fixed per-tensor
    scale; P-Cast Precision review, sections 3 and 5: the static scale S
    multiplies P before the E4M3 cast, KV blocks are visited forward or in
    reverse, and the underflow condition is p * S < 2^-10.
  * FPSAttention article, section 2.2: sliding-tile attention visits only the
    key tiles in a query tile's window, given here as a list per query tile.

Readings where the pages leave a step open:
  * KV tiles of 128 keys; the row max is updated exactly at every tile (no
    lazy threshold), so every probability satisfies p <= 1 and p * S <= S.
  * exp2+cvt P-cast: code = E4M3_RNE_satfinite( fl32( S * exp(x - m) ) ).
  * ExpCast P-cast: z = (x - m) * log2(e) + log2(S) (z includes log2 S, so
    p = 1 maps to the code of S); code = clamp(rne(8 z + 56 + beta), 0, 126).
  * the row sum r_ij is the sum of the DECODED codes (the P that is actually
    multiplied), which makes a constant V come back exactly.
  * a row whose tile list is empty returns 0.
  * the softmax scale defaults to 1/sqrt(128).
"""
from __future__ import annotations

import math

import numpy as np

from .bf16 import round_to_bf16
from . import nvfp4
from .e4m3 import decode, encode

LOG2E = 1.0 / math.log(2.0)
KV_TILE = 128
Q_TILE = 128
QK_BLOCK = 64
V_BLOCK = 128

PCAST_EXP2_CVT = 0
PCAST_EXPCAST = 1
PCAST_FP4 = 2          # 4-bit P with a scale per 16 keys (NVFP4 PV product)


def pcast_codes(x_minus_m: np.ndarray, pcast: int, S: float, beta: float) -> np.ndarray:
    """E4M3 probability codes of logits already reduced by the running max.

    x_minus_m: fp64 natural-log-domain differences x - m (<= 0, may be -inf).
    """
    if pcast == PCAST_EXP2_CVT:
        p = (S * np.exp(x_minus_m)).astype(np.float32)
        return encode(p)
    if pcast == PCAST_EXPCAST:
        z = x_minus_m * LOG2E + math.log2(S)
        c = np.rint(8.0 * z + 56.0 + beta)
        c = np.where(np.isfinite(c), c, 0.0)
        return np.clip(c, 0, 126).astype(np.uint8)
    raise ValueError(f"unknown P-cast mode {pcast}")


def dequant_rows(codes: np.ndarray, scales: np.ndarray, block: int = QK_BLOCK) -> np.ndarray:
    """fp64 values of block-quantised rows: dec(code) * s[row // block] (exact)."""
    T = codes.shape[0]
    s = np.repeat(np.asarray(scales, dtype=np.float64), block)[:T]
    return decode(codes) * s[:, None]


def vtilde(vq: np.ndarray, sv: np.ndarray, mean: np.ndarray, T: int) -> np.ndarray:
    """Dequantised V rows in permuted order: dec(Rq_t) * s_v + mu_blk(t) (fp64 [T,128])."""
    r = decode(vq[:, :T]).T * np.asarray(sv, dtype=np.float64)[None, :]
    mu = np.repeat(np.asarray(mean, dtype=np.float64), V_BLOCK, axis=0)[:T]
    return r + mu


def dense_tile_order(n_tiles: int, reverse: bool) -> list:
    return list(range(n_tiles - 1, -1, -1)) if reverse else list(range(n_tiles))


def tile_list_for_qtile(qt: int, n_tiles: int, reverse: bool, row_ptr=None, col=None) -> list:
    """KV tiles visited by query tile qt, in visiting order.

    Dense: all tiles, ascending (forward) or descending (reverse).
    Sparse: the CSR list col[row_ptr[qt]:row_ptr[qt+1]] as given (forward) or
    backwards (reverse).
    """
    if row_ptr is None:
        return dense_tile_order(n_tiles, reverse)
    lst = [int(c) for c in col[row_ptr[qt]:row_ptr[qt + 1]]]
    return lst[::-1] if reverse else lst


def online_softmax_rows(X: np.ndarray, Vt: np.ndarray, tiles: list, T: int,
                        pcast: int | None, S: float, beta: float,
                        tile: int = KV_TILE, want_weights: bool = False, m_init=None):
    """Blocked online softmax of logit rows X [R, T] against values Vt [T, d].

    m_init [R] (optional): the running max the rows enter with (a split-KV part
    that starts from the exact maximum of the tiles visited before it); by
    default the rows start from -inf.  l and acc always start at zero.

    For each tile in ``tiles`` (visiting order):
      m_new = max(m, max_t x_t);  alpha = exp(m - m_new)
      c_t   = P-cast code of x_t - m_new  (pcast None: no cast, P = exp(x - m_new))
      r     = sum_t dec(c_t);   l = alpha * l + r
      acc   = alpha * acc + sum_t dec(c_t) * V_t
    Returns (acc / l, l, m, weights) with rows of l == 0 giving 0; ``weights``
    (optional) is the effective normalised weight of every key.
    """
    R = X.shape[0]
    d = Vt.shape[1]
    m = np.full(R, -np.inf) if m_init is None else np.array(m_init, dtype=np.float64)
    l = np.zeros(R)
    acc = np.zeros((R, d))
    W = np.zeros((R, T)) if want_weights else None
    for j in tiles:
        lo, hi = j * tile, min((j + 1) * tile, T)
        if lo >= hi:
            continue
        xt = X[:, lo:hi]
        m_new = np.maximum(m, xt.max(axis=1))
        with np.errstate(invalid="ignore"):
            alpha = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        diff = xt - m_new[:, None]
        if pcast is None:
            P = np.exp(diff) * S
        elif pcast == PCAST_FP4:
            P = nvfp4.pcast_fp4(diff)           # 4-bit P, one scale per 16 keys of the tile
        else:
            P = decode(pcast_codes(diff, pcast, S, beta))
        l = alpha * l + P.sum(axis=1)
        acc = alpha[:, None] * acc + P @ Vt[lo:hi]
        if W is not None:
            W *= alpha[:, None]
            W[:, lo:hi] = P
        m = m_new
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
        if W is not None:
            W = np.where(l[:, None] > 0, W / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return out, l, m, W


def split_parts(tiles: list, n_splits: int) -> list:
    """Split-KV (TeleFuser blog, FP8 Sol-Attn mainloop list, long-sequence
    split-KV): the visiting order of a query tile is cut into n_splits
    contiguous parts, part s holding positions [s*n // n_splits, (s+1)*n // n_splits)
    (parts may be empty when the list is short)."""
    n = len(tiles)
    return [tiles[(s * n) // n_splits:((s + 1) * n) // n_splits] for s in range(n_splits)]


def entry_maxima(X: np.ndarray, parts: list, T: int, tile: int = KV_TILE) -> list:
    """Running max with which each part of a split visiting order is entered:
    for part s, the maximum of the logits of every tile in the parts before
    it (-inf for the first part).  Started from it, part s takes the same
    running max at each of its tiles as the unsplit online softmax, so its P
    codes are the unsplit codes."""
    R = X.shape[0]
    out, m = [], np.full(R, -np.inf)
    for part in parts:
        out.append(m.copy())
        for j in part:
            lo, hi = j * tile, min((j + 1) * tile, T)
            if lo < hi:
                m = np.maximum(m, X[:, lo:hi].max(axis=1))
    return out


def lse_merge(outs: list, ls: list, ms: list) -> np.ndarray:
    """Log-sum-exp merge of partial results (same blog passage): part s holds
    out_s = acc_s / l_s, its row sum l_s and running max m_s (natural-log
    units).  With M the largest m_s over parts with l_s > 0 and w_s =
    l_s exp(m_s - M): out = sum_s w_s out_s / sum_s w_s; a row with no key in
    any part gives 0."""
    R = outs[0].shape[0]
    M = np.full(R, -np.inf)
    for l, m in zip(ls, ms):
        M = np.where(l > 0, np.maximum(M, m), M)
    num = np.zeros_like(outs[0])
    den = np.zeros(R)
    for o, l, m in zip(outs, ls, ms):
        with np.errstate(invalid="ignore", over="ignore"):
            w = np.where(l > 0, l * np.exp(np.where(l > 0, m, 0.0) - np.where(np.isfinite(M), M, 0.0)), 0.0)
        num += w[:, None] * o
        den += w
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(den[:, None] > 0, num / np.where(den > 0, den, 1.0)[:, None], 0.0), den


def emulated_attention_head(q_codes, sq, k_codes, sk, vq, sv, mean, T, rows,
                            pcast=PCAST_EXP2_CVT, S=256.0, beta=-0.35,
                            softmax_scale=None, reverse=False, row_ptr=None, col=None,
                            want_weights=False, v_offset=None, n_splits=1, v_hat=None,
                            split_entry_max=False):
    """Emulated FP8 attention for one (batch, head) on selected query rows.

    q_codes [T,128] uint8, sq [ceil(T/64)]  (query order = original order)
    k_codes [T,128] uint8, sk [ceil(T/64)]  (key order = permuted order)
    vq [128, Tpad] uint8, sv [128], mean fp64 [nV,128]  (permuted order)
    rows: query row indices.  Returns (out fp64 of bf16 values [len(rows),128],
    float diagnostics dict).
    v_offset: optional fp32 [128] added to every row that attended at least
    one key, before the bf16 rounding (sequence-mean smoothing of V and the
    bias correction, oracle/smooth.py).
    pcast == PCAST_FP4 (4-bit PV, oracle/nvfp4.py): P is cast to E2M1 with a
    UE4M3 scale per 16 keys, and v_hat (the decoded NVFP4 V, nvfp4.vhat_fp4)
    replaces the E4M3 residual; vq/sv are then ignored.
    n_splits > 1: split-KV — every part of the visiting order (split_parts)
    runs its own online softmax from an empty state, and the parts are merged
    by lse_merge before the offset and the bf16 rounding.  split_entry_max:
    each part instead enters with the running max of the tiles before it
    (entry_maxima), which keeps the unsplit P codes.
    Logits x = scale * sum_c dec(q) sq * dec(k) sk, in fp64 (each product is
    exact; the sum rounds in fp64 only).
    """
    scale = 1.0 / math.sqrt(128.0) if softmax_scale is None or softmax_scale <= 0 else softmax_scale
    rows = np.asarray(rows, dtype=np.int64)
    nT = -(-T // KV_TILE)
    Kd = dequant_rows(k_codes, sk)
    Vt = vtilde(vq, sv, mean, T) if v_hat is None else np.asarray(v_hat, dtype=np.float64)
    out = np.zeros((rows.size, 128))
    l_all = np.zeros(rows.size)
    weights = {} if want_weights else None
    qts = rows // Q_TILE
    for qt in np.unique(qts):
        sel = np.nonzero(qts == qt)[0]
        r = rows[sel]
        Qd = dequant_rows(q_codes[r], sq[r // QK_BLOCK], block=1)
        X = (Qd @ Kd.T) * scale
        tiles = tile_list_for_qtile(int(qt), nT, reverse, row_ptr, col)
        if n_splits == 1:
            o, l, _, W = online_softmax_rows(X, Vt, tiles, T, pcast, S, beta,
                                             want_weights=want_weights)
        else:
            parts = split_parts(tiles, n_splits)
            m0 = entry_maxima(X, parts, T) if split_entry_max else [None] * len(parts)
            res = [online_softmax_rows(X, Vt, part, T, pcast, S, beta, want_weights=want_weights, m_init=mi)
                   for part, mi in zip(parts, m0)]
            o, l = lse_merge([r_[0] for r_ in res], [r_[1] for r_ in res], [r_[2] for r_ in res])
            W = None
            if want_weights:
                W, _ = lse_merge([r_[3] for r_ in res], [r_[1] for r_ in res], [r_[2] for r_ in res])
        out[sel] = o
        l_all[sel] = l
        if want_weights:
            for gi, ri in enumerate(r):
                weights[int(ri)] = W[gi]
    if v_offset is not None:
        out = np.where(l_all[:, None] > 0, out + np.asarray(v_offset, dtype=np.float64)[None, :], out)
    return round_to_bf16(out), dict(l=l_all, weights=weights)


def kept_key_mask(T: int, tiles: list) -> np.ndarray:
    mask = np.zeros(T, dtype=bool)
    for j in tiles:
        mask[j * KV_TILE:min((j + 1) * KV_TILE, T)] = True
    return mask


def exact_attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows,
                         softmax_scale=None, key_mask_for_row=None) -> np.ndarray:
    """Exact softmax(q k^T * scale) v in fp64 for selected rows (no quantisation).

    q, k, v: fp64 [T,128] (k, v in the same key order).  key_mask_for_row:
    optional callable row -> bool mask of the keys that row attends (sparse).
    """
    scale = 1.0 / math.sqrt(128.0) if softmax_scale is None or softmax_scale <= 0 else softmax_scale
    rows = np.asarray(rows, dtype=np.int64)
    X = (q[rows] @ k.T) * scale
    if key_mask_for_row is not None:
        for i, r in enumerate(rows):
            X[i, ~key_mask_for_row(int(r))] = -np.inf
    mx = X.max(axis=1, keepdims=True)
    E = np.exp(X - mx)
    return (E @ v) / E.sum(axis=1, keepdims=True)


def ponly_attention(X: np.ndarray, V: np.ndarray, S: float, reverse: bool, tile: int = 64,
                    pcast: int = PCAST_EXP2_CVT, beta: float = -0.35, rowsum: str = "decoded"):
    """P-only emulation (P-Cast Precision review, section 5): Q, K, V unquantised.

    X: fp64 logits [R, N] (natural-log units), V: fp64 [N, d].  Only the P cast
    is quantised; blocks of ``tile`` keys are visited forward or in reverse.
    rowsum: "decoded" sums the decoded codes (the reading used for the main
    path); "fp32" sums the fp32 probabilities S*exp(x - m) before the cast,
    which is the normalisation under which this emulation reproduces the
    review's MSE table.
    Returns (out [R,d], underflow mask [R,N] of keys cast to code 0).
    """
    N = X.shape[1]
    nT = -(-N // tile)
    order = dense_tile_order(nT, reverse)
    R = X.shape[0]
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    acc = np.zeros((R, V.shape[1]))
    under = np.zeros((R, N), dtype=bool)
    for j in order:
        lo, hi = j * tile, min((j + 1) * tile, N)
        xt = X[:, lo:hi]
        m_new = np.maximum(m, xt.max(axis=1))
        with np.errstate(invalid="ignore"):
            alpha = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        diff = xt - m_new[:, None]
        c = pcast_codes(diff, pcast, S, beta)
        under[:, lo:hi] = c == 0
        P = decode(c)
        if rowsum == "fp32":
            r = (S * np.exp(diff)).astype(np.float32).astype(np.float64).sum(axis=1)
        elif rowsum == "decoded":
            r = P.sum(axis=1)
        else:
            raise ValueError(rowsum)
        l = alpha * l + r
        acc = alpha[:, None] * acc + P @ V[lo:hi]
        m = m_new
    return acc / l[:, None], under

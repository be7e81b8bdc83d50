"""Online V clustering that produces the V-Smooth token permutation (test
infrastructure only).

Follows the VC-Attention news article, section 2 (V-Smooth, first step): a
light clustering of the value tokens of one attention head, on a few
representative dimensions of V, after which the tokens of one cluster are laid
out as one contiguous run, so that the 128-row quantisation blocks of the prep
hold similar rows.  The clusters need not be balanced (only the blocks at
cluster boundaries mix clusters).  The abstract page adds that the clustering
is online and lightweight and that it reorders the value tokens.

Readings (the pages give no formulas):
  * representative dimensions: the r channels of the head with the largest
    max |v| over its T tokens (the channels whose range sets the per-channel
    residual scales); ties go to the lower channel index;
  * similarity is measured on 12-bit fixed-point coordinates: channel d with
    2^E_d <= max_t |v[t,d]| < 2^(E_d+1) is scaled by 2^(11 - E_d) (exact) and
    rounded to the nearest integer, ties to even, so |code| <= 4096; a channel
    of zeros gives codes 0;
  * the clustering is Lloyd's k-means with squared Euclidean distance on those
    codes: seeds are the tokens floor(k T / K), k = 0..K-1; a token joins the
    nearest centroid (ties: the lowest cluster index); a centroid moves to the
    floor of its members' mean code (integer division rounding down), and a
    cluster with no member keeps its centroid; `iters` rounds of (move,
    assign) follow the first assignment;
  * the permutation is the stable sort of the tokens by cluster id: clusters
    in index order, tokens of one cluster in their original order;
    perm[j] = the token placed at position j (the layout the prep's V gather
    reads: V'[j] = V[perm[j]]).
All arithmetic after the fixed-point conversion is exact integer arithmetic.
"""
from __future__ import annotations

import numpy as np

CODE_BITS = 12          # |code| <= 2^CODE_BITS


def representative_dims(v: np.ndarray, r: int) -> np.ndarray:
    """Indices (ascending) of the r channels of v [T, C] with the largest max |v|;
    ties to the lower channel index."""
    amax = np.abs(v).max(axis=0)
    order = sorted(range(v.shape[1]), key=lambda c: (-amax[c], c))
    return np.array(sorted(order[:r]), dtype=np.int64)


def fixed_point_codes(v: np.ndarray, dims: np.ndarray) -> np.ndarray:
    """int64 [T, r] codes: rne(v[:, d] * 2^(11 - E_d)), E_d the exponent of the
    channel's max |v| (an exact power-of-two scaling in fp64)."""
    out = np.zeros((v.shape[0], len(dims)), dtype=np.int64)
    for j, d in enumerate(dims):
        col = v[:, d].astype(np.float64)
        amax = np.abs(col).max()
        if amax == 0.0:
            continue
        E = int(np.floor(np.log2(amax)))
        if 2.0 ** E > amax:          # guard the log2 rounding at exact powers of two
            E -= 1
        elif 2.0 ** (E + 1) <= amax:
            E += 1
        out[:, j] = np.rint(np.ldexp(col, CODE_BITS - 1 - E)).astype(np.int64)
    return out


def assign(codes: np.ndarray, cent: np.ndarray) -> np.ndarray:
    """Nearest centroid of every token (squared Euclidean, ties to the lowest index)."""
    d2 = ((codes[:, None, :] - cent[None, :, :]) ** 2).sum(axis=2)
    return d2.argmin(axis=1)            # argmin returns the first minimum


def move(codes: np.ndarray, labels: np.ndarray, cent: np.ndarray) -> np.ndarray:
    """Centroid update: floor of the member mean; empty clusters stay."""
    new = cent.copy()
    for k in range(cent.shape[0]):
        members = labels == k
        n = int(members.sum())
        if n:
            new[k] = np.floor_divide(codes[members].sum(axis=0), n)
    return new


def kmeans_labels(codes: np.ndarray, n_clusters: int, iters: int):
    """Lloyd's k-means from the evenly spaced seeds; returns (labels, centroids)."""
    T = codes.shape[0]
    seeds = (np.arange(n_clusters, dtype=np.int64) * T) // n_clusters
    cent = codes[seeds].copy()
    labels = assign(codes, cent)
    for _ in range(iters):
        cent = move(codes, labels, cent)
        labels = assign(codes, cent)
    return labels, cent


def stable_perm(labels: np.ndarray) -> np.ndarray:
    """Tokens sorted by cluster id, original order within a cluster."""
    return np.argsort(labels, kind="stable").astype(np.int32)


def cluster_head(v: np.ndarray, n_clusters: int = 32, n_dims: int = 8, iters: int = 4):
    """One head: v [T, 128] (bf16 values as floats) -> (perm int32 [T], labels [T])."""
    dims = representative_dims(v, n_dims)
    codes = fixed_point_codes(v, dims)
    labels, _ = kmeans_labels(codes, n_clusters, iters)
    return stable_perm(labels), labels.astype(np.int32)

"""Pins of the V clustering oracle (oracle/cluster.py).

Checked against exact rational arithmetic (the fixed-point codes), a
brute-force Lloyd iteration written with plain loops on tiny inputs, planted
cluster structure that any correct clustering must recover, the defining
properties of a stable sort, and the effect the VC-Attention news article
(section 2) reports: sorting value tokens by cluster lets the 128-row block
means remove far more of V's energy than the original order does.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import cluster, prep


def _bf(x):
    return obf.round_to_bf16(np.asarray(x, dtype=np.float64))


def test_codes_are_an_exact_power_of_two_scaling():
    rng = np.random.default_rng(31)
    T = 500
    scales = [1.0, 3e-3, 7e4, 2.0 ** -20, 1.0]
    v = np.stack([_bf(rng.standard_normal(T) * s) for s in scales], axis=1)
    v[:, 4] = 0.0                                       # a channel of zeros
    v[7, 0] = 4.0                                       # exact power-of-two maximum
    codes = cluster.fixed_point_codes(v, np.arange(5))
    assert np.all(codes[:, 4] == 0)
    for d in range(4):
        amax = np.max(np.abs(v[:, d]))
        E = 0
        while Fraction(2) ** (E + 1) <= Fraction(float(amax)):
            E += 1
        while Fraction(2) ** E > Fraction(float(amax)):
            E -= 1
        unit = Fraction(2) ** (E - 11)
        for t in range(T):
            exact = Fraction(float(v[t, d])) / unit
            assert abs(exact - codes[t, d]) <= Fraction(1, 2)
            if abs(exact - codes[t, d]) == Fraction(1, 2):
                assert codes[t, d] % 2 == 0              # ties to even
        assert 2048 <= np.max(np.abs(codes[:, d])) <= 4096
    assert codes[7, 0] == 2048
    # a halfway value rounds to the even neighbour: 2.5 and 3.5 units
    w = np.zeros((3, 1))
    w[:, 0] = [1.0, 2.5 * 2.0 ** -11, 3.5 * 2.0 ** -11]
    assert cluster.fixed_point_codes(w, np.array([0]))[:, 0].tolist() == [2048, 2, 4]


def test_representative_dims_are_the_widest_channels():
    v = np.zeros((4, 10))
    amax = [1, 5, 3, 5, 0, 2, 5, 4, 1, 0.5]
    for c, a in enumerate(amax):
        v[c % 4, c] = -a if c % 2 else a
    assert cluster.representative_dims(v, 3).tolist() == [1, 3, 6]       # the three 5s
    assert cluster.representative_dims(v, 5).tolist() == [1, 2, 3, 6, 7]
    assert cluster.representative_dims(v, 1).tolist() == [1]             # tie: lowest channel


def _lloyd_by_loops(codes, K, iters):
    T, r = len(codes), len(codes[0])
    cent = [list(codes[(k * T) // K]) for k in range(K)]

    def nearest(x):
        best, arg = None, 0
        for k in range(K):
            d = sum((x[j] - cent[k][j]) ** 2 for j in range(r))
            if best is None or d < best:
                best, arg = d, k
        return arg

    labels = [nearest(x) for x in codes]
    for _ in range(iters):
        for k in range(K):
            members = [codes[t] for t in range(T) if labels[t] == k]
            if members:
                cent[k] = [sum(m[j] for m in members) // len(members) for j in range(r)]
        labels = [nearest(x) for x in codes]
    return labels


@pytest.mark.parametrize("T,K,r,iters", [(40, 5, 3, 3), (61, 7, 2, 0), (33, 4, 4, 6), (9, 12, 1, 2)])
def test_kmeans_matches_a_brute_force_lloyd_iteration(T, K, r, iters):
    rng = np.random.default_rng(32 + T)
    codes = rng.integers(-4096, 4097, (T, r))
    codes[rng.integers(0, T, 5)] = codes[0]              # repeated points make ties
    labels, _ = cluster.kmeans_labels(codes.astype(np.int64), K, iters)
    assert labels.tolist() == _lloyd_by_loops([list(map(int, x)) for x in codes], K, iters)


def test_contiguous_clusters_are_recovered_exactly():
    # eight well-separated groups laid out as runs (as neighbouring video tokens are)
    rng = np.random.default_rng(33)
    T, G = 2000, 8
    centres = 6 * rng.standard_normal((G, 128))
    truth = np.repeat(np.arange(G), T // G)
    v = _bf(centres[truth] + 0.1 * rng.standard_normal((T, 128)))
    perm, labels = cluster.cluster_head(v, n_clusters=G, n_dims=8, iters=3)
    assert labels.tolist() == truth.tolist()
    assert perm.tolist() == list(range(T))


def test_more_clusters_than_structure_gives_pure_clusters():
    rng = np.random.default_rng(34)
    T, G = 3000, 6
    centres = 6 * rng.standard_normal((G, 128))
    truth = rng.integers(0, G, T)
    v = _bf(centres[truth] + 0.1 * rng.standard_normal((T, 128)))
    perm, labels = cluster.cluster_head(v, n_clusters=24, n_dims=8, iters=4)
    for k in np.unique(labels):
        assert len(np.unique(truth[labels == k])) == 1           # no cluster mixes groups
    # the permutation lays every cluster out as one contiguous run
    runs = labels[perm]
    assert np.all(np.diff(runs) >= 0)


def test_perm_is_a_stable_sort_by_cluster_id():
    rng = np.random.default_rng(35)
    labels = rng.integers(0, 9, 777)
    perm = cluster.stable_perm(labels)
    assert sorted(perm.tolist()) == list(range(777))
    for k in range(9):
        pos = perm[labels[perm] == k]
        assert np.all(np.diff(pos) > 0)                    # original order inside a cluster
    assert np.all(np.diff(labels[perm]) >= 0)


def test_degenerate_cases():
    rng = np.random.default_rng(36)
    v = _bf(rng.standard_normal((300, 128)))
    perm, labels = cluster.cluster_head(v, n_clusters=1)
    assert perm.tolist() == list(range(300)) and np.all(labels == 0)
    const = np.full((200, 128), 1.5)
    perm, labels = cluster.cluster_head(const, n_clusters=16)
    assert perm.tolist() == list(range(200)) and np.all(labels == 0)    # all ties -> cluster 0
    zero = np.zeros((50, 128))
    perm, labels = cluster.cluster_head(zero, n_clusters=4)
    assert perm.tolist() == list(range(50))
    few = _bf(rng.standard_normal((5, 128)) * 3)
    perm, labels = cluster.cluster_head(few, n_clusters=8, iters=2)
    assert sorted(perm.tolist()) == list(range(5))
    assert len(np.unique(labels)) == 5                     # every distinct token its own cluster


def test_cluster_order_lets_block_means_remove_energy():
    # VC-Attention news article, section 2: block means remove 8 % of V's energy in the
    # original token order and 36 % after sorting tokens by value cluster (Wan2.2 heads)
    rng = np.random.default_rng(37)
    T = 16384                      # 128 blocks: the 31 cluster boundaries mix few of them
    cid = rng.integers(0, 16, T)
    centres = 4 * rng.standard_normal((16, 128))
    vh = centres[cid] + 0.5 * rng.standard_normal((T, 128))
    vh[rng.permutation(T)[: T // 200]] *= 20.0
    v = _bf(vh)
    energy = np.sum(v ** 2)

    def removed(perm):
        out = prep.prep_v_head(v, perm, vsmooth=True)
        return 1 - np.sum(out["resid"].astype(np.float64) ** 2) / energy

    perm, _ = cluster.cluster_head(v)
    r_orig, r_truth, r_clustered = removed(None), removed(np.argsort(cid, kind="stable")), removed(perm)
    assert r_orig < 0.1
    assert r_clustered > 0.75 * r_truth and r_clustered > 5 * r_orig

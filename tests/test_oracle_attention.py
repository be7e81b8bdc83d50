"""Pins of the oracle's stage 2: online softmax, P-cast study, decomposition.

Checked against brute-force direct softmax, the special cases of the method
(constant V, zero queries), the algebraic error decomposition, and the
P-Cast Precision review's Table I / MSE table / theorems.
"""
import math
import os

import numpy as np
import pytest

from oracle import attention as A
from oracle import closed_forms as cf
from oracle import prep
from oracle.bf16 import round_to_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _direct_softmax(X, V, keep):
    Xm = np.where(keep, X, -np.inf)
    E = np.exp(Xm - Xm.max(axis=1, keepdims=True))
    return (E @ V) / E.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129, 300])
def test_blocked_online_softmax_equals_direct_softmax(T):
    rng = np.random.default_rng(T)
    X = rng.standard_normal((7, T)) * 3
    V = rng.standard_normal((T, 16))
    nT = -(-T // 128)
    for tiles in (list(range(nT)), list(range(nT))[::-1]):
        out, _, _, _ = A.online_softmax_rows(X, V, tiles, T, None, 1.0, 0.0)
        ref = _direct_softmax(X, V, np.ones(T, dtype=bool))
        assert np.max(np.abs(out - ref)) <= 1e-13 * max(1.0, np.max(np.abs(ref)))
    # a random sparse tile subset visited in random order
    sub = sorted(rng.choice(nT, size=max(1, nT // 2), replace=False).tolist())
    rng.shuffle(sub)
    out, _, _, _ = A.online_softmax_rows(X, V, sub, T, None, 1.0, 0.0)
    keep = A.kept_key_mask(T, sub)
    assert np.max(np.abs(out - _direct_softmax(X, V, keep))) <= 1e-13 * max(1.0, np.max(np.abs(V)))


def test_tile_lists():
    assert A.tile_list_for_qtile(0, 4, False) == [0, 1, 2, 3]
    assert A.tile_list_for_qtile(0, 4, True) == [3, 2, 1, 0]
    rp = np.array([0, 2, 2, 5])
    col = np.array([1, 3, 0, 1, 2])
    assert A.tile_list_for_qtile(0, 4, False, rp, col) == [1, 3]
    assert A.tile_list_for_qtile(1, 4, True, rp, col) == []
    assert A.tile_list_for_qtile(2, 4, True, rp, col) == [2, 1, 0]


def _prep_head(rng, T, v=None, q=None, vsmooth=True):
    from oracle.bf16 import round_to_bf16 as r16
    q = r16(rng.standard_normal((T, 128))) if q is None else q
    k = r16(rng.standard_normal((T, 128)))
    v = r16(rng.standard_normal((T, 128))) if v is None else v
    qc, sq = prep.quantize_qk_head(q)
    kc, sk = prep.quantize_qk_head(k)
    pv = prep.prep_v_head(v, None, vsmooth)
    return q, k, v, qc, sq, kc, sk, pv


@pytest.mark.parametrize("pcast", [A.PCAST_EXP2_CVT, A.PCAST_EXPCAST])
def test_constant_v_is_preserved_exactly(pcast):
    rng = np.random.default_rng(11)
    T = 333
    v = np.full((T, 128), -2.375)
    _, _, _, qc, sq, kc, sk, pv = _prep_head(rng, T, v=v, vsmooth=True)
    out, _ = A.emulated_attention_head(qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T,
                                       rows=np.arange(T), pcast=pcast)
    assert np.all(out == -2.375)


def test_zero_queries_give_the_mean_of_dequantised_v():
    rng = np.random.default_rng(12)
    T = 200
    _, _, _, qc, sq, kc, sk, pv = _prep_head(rng, T, q=np.zeros((T, 128)))
    out, _ = A.emulated_attention_head(qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T,
                                       rows=np.arange(0, T, 7))
    vt = A.vtilde(pv["vq"], pv["sv"], pv["mean"], T)
    assert np.array_equal(out, np.broadcast_to(round_to_bf16(vt.mean(axis=0)), out.shape))


def test_empty_tile_list_gives_zero():
    rng = np.random.default_rng(13)
    T = 256
    _, _, _, qc, sq, kc, sk, pv = _prep_head(rng, T)
    rp = np.array([0, 0, 1])
    col = np.array([1])
    out, _ = A.emulated_attention_head(qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T,
                                       rows=np.arange(T), row_ptr=rp, col=col)
    assert np.all(out[:128] == 0) and np.any(out[128:] != 0)


@pytest.mark.parametrize("pcast", [A.PCAST_EXP2_CVT, A.PCAST_EXPCAST])
@pytest.mark.parametrize("vsmooth", [False, True])
def test_emulation_is_close_to_exact_attention(pcast, vsmooth):
    rng = np.random.default_rng(14)
    T = 1024
    q, k, v, qc, sq, kc, sk, pv = _prep_head(rng, T, vsmooth=vsmooth)
    rows = np.arange(0, T, 3)
    out, _ = A.emulated_attention_head(qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T,
                                       rows=rows, pcast=pcast)
    ref = A.exact_attention_rows(q, k, v, rows)
    cos = np.sum(out * ref) / np.linalg.norm(out) / np.linalg.norm(ref)
    assert cos > 0.99


def test_forward_and_reverse_agree_without_quantisation():
    rng = np.random.default_rng(15)
    X = rng.standard_normal((5, 700)) * 4
    V = rng.standard_normal((700, 8))
    a, _, _, _ = A.online_softmax_rows(X, V, [0, 1, 2, 3, 4, 5], 700, None, 1.0, 0.0)
    b, _, _, _ = A.online_softmax_rows(X, V, [5, 4, 3, 2, 1, 0], 700, None, 1.0, 0.0)
    assert np.max(np.abs(a - b)) < 1e-13


def test_error_decomposition_identity():
    # VC-Attention: O - Oq = (P - Pq) V + Pq (V - Vq)
    rng = np.random.default_rng(16)
    T = 512
    q, k, v, qc, sq, kc, sk, pv = _prep_head(rng, T, vsmooth=True)
    rows = np.arange(0, T, 5)
    _, diag = A.emulated_attention_head(qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T,
                                        rows=rows, want_weights=True)
    Pq = np.stack([diag["weights"][int(r)] for r in rows])
    Qd = A.dequant_rows(qc, sq)
    Kd = A.dequant_rows(kc, sk)
    X = (Qd[rows] @ Kd.T) / math.sqrt(128)
    P = np.exp(X - X.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    Vq = A.vtilde(pv["vq"], pv["sv"], pv["mean"], T)
    total, pterm, vterm = cf.decomposition(P, Pq, v, Vq)
    assert np.max(np.abs(total - (pterm + vterm))) < 1e-12
    assert np.allclose(Pq.sum(axis=1), 1.0, atol=1e-12)


def _sink_logits(rng, R, N, delta, k=4):
    X = rng.standard_normal((R, N))
    X[:, :k] += delta
    return X


def test_delta4_matches_the_page():
    # Proposition 1 note: delta_4 ~= 1.03 (not sqrt(2 ln 4) ~= 1.67)
    assert abs(cf.delta_k(4) - 1.03) < 0.005
    assert abs(cf.underflow_threshold(1.0) - 6.93) < 0.005
    assert abs(cf.underflow_threshold(256.0) - 10 * math.log(2) - 8 * math.log(2)) < 1e-12
    assert abs(18 * math.log(2) - 12.48) < 0.005


def test_p_collapse_table1():
    """Monte Carlo of the oracle's P-only emulation and the averaged closed form vs Table I.

    Tolerance 3 points absolute: the page's own sampling noise is unknown and the
    oracle's Monte Carlo at 2048 rows has a standard error of about 0.5 point;
    an error in the underflow threshold (e.g. 2^-9 for 2^-10, or a dropped ln S)
    moves these fractions by 10-25 points.
    """
    rng = np.random.default_rng(17)
    N, R = 4096, 2048
    V = np.ones((N, 1))
    for row in _load("p_collapse_table1.txt"):
        delta, f1, f256, mass, loss = (float(x) for x in row)
        X = _sink_logits(rng, R, N, delta)
        _, u1 = A.ponly_attention(X, V, 1.0, reverse=False, tile=64)
        _, u256 = A.ponly_attention(X, V, 256.0, reverse=False, tile=64)
        mc1 = 100 * u1[:, 4:].mean()
        mc256 = 100 * u256[:, 4:].mean()
        E = np.exp(X - X.max(axis=1, keepdims=True))
        mc_mass = 100 * np.mean(E[:, 4:].sum(axis=1) / E.sum(axis=1))
        assert abs(mc1 - f1) <= 3.0, (delta, mc1, f1)
        assert abs(mc256 - f256) <= 3.0, (delta, mc256, f256)
        assert abs(mc_mass - mass) <= 3.0, (delta, mc_mass, mass)
        assert abs(mc1 * mc_mass / 100 - loss) <= 3.0, (delta, mc1 * mc_mass / 100, loss)
        # closed form of Proposition 1, with the sink max averaged over its law
        assert abs(100 * cf.underflow_fraction_averaged(delta, 1.0) - f1) <= 3.0
        assert abs(100 * cf.underflow_fraction_averaged(delta, 256.0) - f256) <= 3.0
        # the printed plug-in form is coarser (it ignores the spread of the sink max)
        assert abs(100 * cf.underflow_fraction_plugin(delta, 1.0) - f1) <= 6.0
        # per row, underflow is exactly "logit below m - 10 ln 2 - ln S" (up to ties)
        m = X.max(axis=1, keepdims=True)
        pred = X[:, 4:] < m - cf.underflow_threshold(1.0)
        assert np.mean(pred != u1[:, 4:]) < 1e-3


def test_reverse_order_with_s256_has_no_underflow_before_the_sinks():
    # Theorem 4: reverse + S=256 keeps every non-sink block above the round-to-zero edge
    rng = np.random.default_rng(18)
    N, R = 4096, 512
    for delta in (5.0, 7.0, 10.0):
        X = _sink_logits(rng, R, N, delta)
        _, u = A.ponly_attention(X, np.ones((N, 1)), 256.0, reverse=True, tile=64)
        assert u[:, 64:].sum() == 0
        assert cf.reverse_order_bound(X[:, 64:].max()) < 1e-12


def test_p_cast_mse_table():
    """P-only MSE vs the review's table (Delta = 7): orderings, and levels within 35 %.

    MSE is averaged over three independent (logits, V) draws of 256 rows; the
    draw-to-draw spread of a single draw is about 15 %.
    """
    rng = np.random.default_rng(19)
    table = {r[0]: [float(x) for x in r[1:]] for r in _load("p_cast_mse.txt")}
    cfgs = {"fwd_S1": (1.0, False), "rev_S1": (1.0, True), "fwd_S448": (448.0, False),
            "fwd_S256": (256.0, False), "rev_S256": (256.0, True)}
    ratios = []
    for ni, N in enumerate((4096, 8192)):
        mse = {name: 0.0 for name in cfgs}
        for _ in range(3):
            X = _sink_logits(rng, 256, N, 7.0)
            V = rng.standard_normal((N, 128))
            E = np.exp(X - X.max(axis=1, keepdims=True))
            O = (E @ V) / E.sum(axis=1, keepdims=True)
            for name, (S, rev) in cfgs.items():
                o, _ = A.ponly_attention(X, V, S, rev, tile=64, rowsum="fp32")
                mse[name] += np.mean((o - O) ** 2) * 1e5 / 3
        for name in cfgs:
            assert abs(mse[name] / table[name][ni] - 1) < 0.35, (N, name, mse[name], table[name][ni])
        best = min(mse.values())
        assert mse["fwd_S1"] > 2.5 * best
        for name in ("rev_S1", "fwd_S448", "fwd_S256", "rev_S256"):
            assert mse[name] < 1.25 * best
        assert mse["fwd_S256"] <= mse["fwd_S448"]
        ratios.append(mse["fwd_S1"] / best)
    assert ratios[1] > ratios[0]            # the forward S=1 penalty grows with N


# ---- split-KV with a log-sum-exp merge (TeleFuser blog, FP8 Sol-Attn mainloop,
# long-sequence split-KV)

def test_split_parts_cover_the_visiting_order_once():
    tiles = [7, 3, 9, 1, 4]
    for S in (1, 2, 3, 5, 8):
        parts = A.split_parts(tiles, S)
        assert len(parts) == S
        assert sum(parts, []) == tiles                      # contiguous, in order, each once
        assert max(len(p) for p in parts) - min(len(p) for p in parts) <= 1
    assert A.split_parts([], 3) == [[], [], []]


@pytest.mark.parametrize("T,S", [(300, 2), (1000, 3), (1000, 8), (129, 4), (64, 3)])
def test_split_merge_without_quantisation_equals_direct_softmax(T, S):
    # with the P cast switched off the split is exact: every part carries its own
    # running max, and the log-sum-exp merge must give the direct softmax back
    rng = np.random.default_rng(40 + S)
    X = rng.standard_normal((6, T)) * 4
    X[2, 5:9] += 30.0                                       # a row dominated by a few keys
    V = rng.standard_normal((T, 16))
    nT = -(-T // 128)
    for tiles in (list(range(nT)), list(range(nT))[::-1]):
        res = [A.online_softmax_rows(X, V, part, T, None, 256.0, 0.0) for part in A.split_parts(tiles, S)]
        out, den = A.lse_merge([r[0] for r in res], [r[1] for r in res], [r[2] for r in res])
        ref = _direct_softmax(X, V, np.ones(T, dtype=bool))
        assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
        # the merged denominator is the full row sum in the frame of the largest max
        full = A.online_softmax_rows(X, V, tiles, T, None, 256.0, 0.0)
        assert np.allclose(den, full[1], rtol=1e-12)


@pytest.mark.parametrize("pcast", [A.PCAST_EXP2_CVT, A.PCAST_EXPCAST])
@pytest.mark.parametrize("T", [1000, 777])
def test_split_entering_with_the_running_max_keeps_the_unsplit_codes(pcast, T):
    # a part that enters with the exact maximum of the tiles before it takes the
    # unsplit running max at every one of its tiles, so it casts the unsplit P
    # codes: the merged weights of every key and the merged output equal the
    # unsplit ones up to fp64 rounding order.  Parts that start from -inf cast
    # against their own max and differ by whole code steps.
    rng = np.random.default_rng(43 + T)
    X = rng.standard_normal((8, T)) * 3
    X[3, 700:705] += 12.0                                   # a late maximum moves the frame
    X[5, 10:12] += 9.0                                      # an early one dominates
    V = rng.standard_normal((T, 16))
    nT = -(-T // 128)
    for tiles in (list(range(nT)), list(range(nT))[::-1], [5, 0, 3, 1, 4, 2]):
        full = A.online_softmax_rows(X, V, tiles, T, pcast, 256.0, -0.35, want_weights=True)
        for S in (2, 3, 4):
            parts = A.split_parts(tiles, S)
            m0 = A.entry_maxima(X, parts, T)
            res = [A.online_softmax_rows(X, V, pt, T, pcast, 256.0, -0.35, want_weights=True, m_init=mi)
                   for pt, mi in zip(parts, m0)]
            out, den = A.lse_merge([r[0] for r in res], [r[1] for r in res], [r[2] for r in res])
            W, _ = A.lse_merge([r[3] for r in res], [r[1] for r in res], [r[2] for r in res])
            assert np.max(np.abs(out - full[0])) <= 1e-12 * np.max(np.abs(full[0]))
            assert np.allclose(W, full[3], rtol=1e-12, atol=0.0)
            assert np.allclose(den, full[1], rtol=1e-12)
            own = [A.online_softmax_rows(X, V, pt, T, pcast, 256.0, -0.35, want_weights=True) for pt in parts]
            W_own, _ = A.lse_merge([r[3] for r in own], [r[1] for r in own], [r[2] for r in own])
            assert not np.allclose(W_own, full[3], rtol=1e-6, atol=0.0)
    # through the head-level entry point: bf16 outputs equal the unsplit ones
    q, k, v, qc, sq, kc, sk, pv = _prep_head(rng, T)
    args = (qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T)
    rows = np.arange(T)
    a, _ = A.emulated_attention_head(*args, rows=rows, pcast=pcast)
    b, _ = A.emulated_attention_head(*args, rows=rows, pcast=pcast, n_splits=4, split_entry_max=True)
    assert np.mean(a == b) > 0.9999 and np.max(np.abs(a - b)) <= 2.0 ** -7 * np.max(np.abs(a))
    c, _ = A.emulated_attention_head(*args, rows=rows, pcast=pcast, n_splits=4)
    assert np.mean(a == c) < 0.5                             # parts from -inf: other codes


def test_split_with_single_nonempty_part_equals_unsplit():
    rng = np.random.default_rng(41)
    T = 384
    _, _, _, qc, sq, kc, sk, pv = _prep_head(rng, T)
    rp = np.array([0, 1, 1, 2])                              # one tile, none, one tile
    col = np.array([2, 0])
    args = (qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T)
    a, _ = A.emulated_attention_head(*args, rows=np.arange(T), row_ptr=rp, col=col)
    b, _ = A.emulated_attention_head(*args, rows=np.arange(T), row_ptr=rp, col=col, n_splits=4)
    assert np.array_equal(a, b)
    assert np.all(b[128:256] == 0)                           # the empty list stays 0


@pytest.mark.parametrize("pcast", [A.PCAST_EXP2_CVT, A.PCAST_EXPCAST])
def test_split_preserves_constant_v_and_stays_close(pcast):
    rng = np.random.default_rng(42)
    T = 1000
    v = np.full((T, 128), 1.625)
    _, _, _, qc, sq, kc, sk, pv = _prep_head(rng, T, v=v)
    out, _ = A.emulated_attention_head(qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T,
                                       rows=np.arange(T), pcast=pcast, n_splits=3)
    assert np.all(out == 1.625)
    q, k, v, qc, sq, kc, sk, pv = _prep_head(rng, T)
    rows = np.arange(0, T, 5)
    args = (qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T)
    ref = A.exact_attention_rows(q, k, v, rows)
    e1 = np.linalg.norm(A.emulated_attention_head(*args, rows=rows, pcast=pcast)[0] - ref)
    e4 = np.linalg.norm(A.emulated_attention_head(*args, rows=rows, pcast=pcast, n_splits=4)[0] - ref)
    assert e4 <= 1.5 * e1                                    # each part quantises against its own max

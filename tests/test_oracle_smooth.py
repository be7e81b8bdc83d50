"""Pins of the sequence-mean smoothing oracle (oracle/smooth.py).

Checked against exact rational arithmetic, the softmax shift invariance and
the unit row sum the TeleFuser blog (section "Diffusion precision guards")
states, and a closed case: with all logits equal every key gets the same
weight, so the corrected output must be the plain mean of V.
"""
from fractions import Fraction

import numpy as np

from oracle import attention as A
from oracle import prep, smooth
from oracle.bf16 import round_to_bf16


def _bf(x):
    return round_to_bf16(np.asarray(x, dtype=np.float64))


def test_round_fraction_to_f32_is_nearest_even():
    rng = np.random.default_rng(21)
    for _ in range(400):
        q = Fraction(int(rng.integers(-10**12, 10**12)), int(rng.integers(1, 10**9)))
        got = smooth.round_fraction_to_f32(q)
        lo = np.nextafter(got, np.float32(-np.inf))
        hi = np.nextafter(got, np.float32(np.inf))
        d = abs(Fraction(float(got)) - q)
        assert d <= abs(Fraction(float(lo)) - q) and d <= abs(Fraction(float(hi)) - q)
    # ties go to the even mantissa
    one = np.float32(1.0)
    half_up = (Fraction(1) + Fraction(float(np.nextafter(one, np.float32(2))))) / 2
    assert smooth.round_fraction_to_f32(half_up) == one
    # values already in fp32 come back unchanged
    for v in (np.float32(3.25), np.float32(-1e-20), np.float32(6.1e37)):
        assert smooth.round_fraction_to_f32(Fraction(float(v))) == v


def test_seq_mean_is_the_exact_mean_rounded_once():
    rng = np.random.default_rng(22)
    for T, spread in ((37, 1), (300, 6), (128, 30)):
        x = _bf(rng.standard_normal((T, 8)) * 10.0 ** rng.uniform(-spread, spread, (T, 8)))
        got = smooth.seq_mean_f32(x)
        for c in range(8):
            exact = sum(Fraction(float(v)) for v in x[:, c]) / T
            assert got[c] == smooth.round_fraction_to_f32(exact), (T, c)


def test_k_centering_leaves_exact_attention_unchanged():
    rng = np.random.default_rng(23)
    T = 200
    q = _bf(rng.standard_normal((T, 128)))
    k = _bf(rng.standard_normal((T, 128)) + 3 * rng.standard_normal((1, 128)))
    v = _bf(rng.standard_normal((T, 128)))
    kbar = smooth.seq_mean_f32(k)
    rows = np.arange(T)
    a = A.exact_attention_rows(q, k, v, rows)
    # the exact shift adds the same constant to every logit of a row
    b = A.exact_attention_rows(q, k - kbar.astype(np.float64)[None, :], v, rows)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))
    # the fp32 centring moves each entry by at most half an fp32 step
    c = A.exact_attention_rows(q, smooth.center(k, kbar), v, rows)
    assert np.max(np.abs(a - c)) <= 1e-6 * np.max(np.abs(a))


def test_v_centering_plus_mean_restores_exact_attention():
    rng = np.random.default_rng(24)
    T = 200
    q = _bf(rng.standard_normal((T, 128)))
    k = _bf(rng.standard_normal((T, 128)))
    v = _bf(rng.standard_normal((T, 128)) + 5)
    vbar = smooth.seq_mean_f32(v)
    rows = np.arange(T)
    a = A.exact_attention_rows(q, k, v, rows)
    b = A.exact_attention_rows(q, k, v - vbar.astype(np.float64), rows) + vbar.astype(np.float64)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))


def test_bias_correction_restores_the_mean_under_uniform_weights():
    # Q = 0: every logit is 0, every P code is the code of S, every key gets
    # the same weight; the output is mean(Vhat') + vbar - b = mean(V') + vbar
    rng = np.random.default_rng(25)
    T = 333
    q = np.zeros((T, 128))
    k = _bf(rng.standard_normal((T, 128)))
    v = _bf(rng.standard_normal((T, 128)) * 2 + rng.standard_normal((1, 128)) * 4)
    perm = rng.permutation(T)
    for vsmooth in (False, True):
        vbar = smooth.seq_mean_f32(v)
        qc, sq = prep.quantize_qk_head(q)
        kc, sk = prep.quantize_qk_head(k[perm])
        r = prep.prep_v_head(v, perm, vsmooth, vbar=vbar)
        b = smooth.v_bias(r["vq"], r["sv"], r["mean"], r["vprime"])
        off = vbar.astype(np.float64) - b
        rows = np.arange(0, T, 5)
        o, _ = A.emulated_attention_head(qc, sq, kc, sk, r["vq"], r["sv"], r["mean"], T, rows,
                                         v_offset=off)
        want = v.mean(axis=0)
        tol = np.abs(want) * 2.0 ** -8 + 1e-5       # one bf16 rounding of the output
        assert np.all(np.abs(o - want[None, :]) <= tol[None, :]), vsmooth
        # without the correction the quantisation bias stays in the output
        o2, _ = A.emulated_attention_head(qc, sq, kc, sk, r["vq"], r["sv"], r["mean"], T, rows,
                                          v_offset=vbar.astype(np.float64))
        assert np.abs(o2 - want[None, :]).mean() >= np.abs(o - want[None, :]).mean()


def test_k_smoothing_reduces_the_error_on_channel_offsets():
    # the Wan2.1-shaped recipe: constant offsets on 4 channels dominate the K
    # block maxima; centring K removes them before the 64-token quantisation
    rng = np.random.default_rng(26)
    T = 640
    ch = rng.choice(128, 4, replace=False)
    q = rng.standard_normal((T, 128))
    k = rng.standard_normal((T, 128))
    q[:, ch] += rng.normal(0, 3, 4)
    k[:, ch] += rng.normal(0, 3, 4)
    q, k, v = _bf(q), _bf(k), _bf(rng.standard_normal((T, 128)))
    rows = np.arange(0, T, 3)
    ex = A.exact_attention_rows(q, k, v, rows)
    errs = []
    for smoothk in (False, True):
        kk = smooth.center(k, smooth.seq_mean_f32(k)) if smoothk else k
        qc, sq = prep.quantize_qk_head(q)
        kc, sk = prep.quantize_qk_head(kk)
        r = prep.prep_v_head(v, None, True)
        o, _ = A.emulated_attention_head(qc, sq, kc, sk, r["vq"], r["sv"], r["mean"], T, rows)
        errs.append(np.linalg.norm(o - ex) / np.linalg.norm(ex))
    assert errs[1] < 0.9 * errs[0], errs


def test_block_means_of_centred_fp32_rows_are_exact():
    rng = np.random.default_rng(27)
    v = _bf(rng.standard_normal((200, 128)) * 3 + 7)
    vp = smooth.center(v, smooth.seq_mean_f32(v))     # fp32 values, 24-bit significands
    mu = prep.block_means(vp)
    for j, lo in enumerate(range(0, 200, 128)):
        blk = vp[lo:lo + 128]
        for c in (0, 5, 77, 127):
            exact = sum(Fraction(float(x)) for x in blk[:, c]) / blk.shape[0]
            assert mu[j, c] == prep._round_fraction_to_bf16(exact)

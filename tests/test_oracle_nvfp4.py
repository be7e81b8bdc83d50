"""Pins of the 4-bit (NVFP4) PV oracle (oracle/nvfp4.py).

Checked against a brute-force nearest-value search over the E2M1 table,
exact rational bounds of the block quantisation, the special cases the
method fixes (a constant V returns exactly under V-Smooth; equal logits give
the plain mean of the decoded V), and closeness to exact attention.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention as A
from oracle import e4m3
from oracle import nvfp4 as N
from oracle import prep
from oracle.bf16 import round_to_bf16


def _brute_e2m1(x: float) -> int:
    best, code = None, 0
    for c in range(8):
        d = abs(abs(x) - N.E2M1_VALUES[c])
        if best is None or d < best or (d == best and c % 2 == 0):
            best, code = d, c
    if abs(x) >= 6:
        code = 7
    return code | (8 if np.signbit(x) else 0)


def test_e2m1_table_and_encoder():
    assert N.e2m1_decode(np.arange(16)).tolist() == [0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6]
    grid = set()
    for v in N.E2M1_VALUES:
        for d in (0.0, 1e-7, -1e-7):
            grid.update({v + d, -(v + d)})
    for m in (N.E2M1_VALUES[:-1] + N.E2M1_VALUES[1:]) / 2:    # every midpoint and its neighbours
        for d in (0.0, 1e-6, -1e-6):
            grid.update({m + d, -(m + d)})
    grid.update({7.0, 100.0, -6.5, 1e-30, -1e-30, 0.1, 3.3})
    xs = np.array(sorted(grid), dtype=np.float32)
    got = N.e2m1_encode(xs)
    for x, c in zip(xs, got):
        assert c == _brute_e2m1(float(x)), (x, c)
    # encode o decode is the identity on the table
    assert np.array_equal(N.e2m1_encode(N.e2m1_decode(np.arange(16))), np.arange(16))


def test_residual_block_quantisation_bounds():
    rng = np.random.default_rng(50)
    T = 300                                       # a ragged last 16-token block (300 = 18*16 + 12)
    resid = (rng.standard_normal((T, 128)) * np.exp(rng.uniform(-3, 3, (1, 128)))).astype(np.float32)
    resid[:, 5] = 0.0                             # a channel of zeros
    codes, sfc, s_c, amax = N.quantize_residual(resid)
    assert s_c[5] == 0 and np.all(codes[5] == 0) and np.all(sfc[5] == 0)
    assert codes.shape == (128, 384) and np.all(codes[:, T:] == 0)
    for c in (0, 1, 77):
        # the channel maximum maps to the top of the two-level range: its block scale is 448
        bmax = int(np.argmax(np.abs(resid[:, c]))) // 16
        assert e4m3.decode(sfc[c, bmax]) == 448.0
        for b in range(-(-T // 16)):
            s, e = 16 * b, min(16 * b + 16, T)
            sfv = Fraction(float(e4m3.decode(sfc[c, b])))
            dec = [Fraction(float(N.e2m1_decode(q))) * sfv * Fraction(float(s_c[c])) for q in codes[c, s:e]]
            for x, xh in zip(resid[s:e, c], dec):
                # the E2M1 step at the block's top binade is 2 units of sf * s_c: error <= half of it,
                # plus the small mismatch between 1/G and s_c
                assert abs(Fraction(float(x)) - xh) <= sfv * Fraction(float(s_c[c])) * Fraction(1001, 1000)


def test_constant_v_is_exact_under_v_smooth():
    rng = np.random.default_rng(51)
    T = 333
    v = np.full((T, 128), 2.75)
    out = N.prep_v_head_fp4(v, None, vsmooth=True)
    assert np.all(out["v4"] == 0) and np.all(out["sc"] == 0)
    vh = N.vhat_fp4(out["v4"], out["sf"], out["sc"], out["mean"], T)
    assert np.all(vh == 2.75)
    q = round_to_bf16(rng.standard_normal((T, 128)))
    k = round_to_bf16(rng.standard_normal((T, 128)))
    qc, sq = prep.quantize_qk_head(q)
    kc, sk = prep.quantize_qk_head(k)
    o, _ = A.emulated_attention_head(qc, sq, kc, sk, None, None, out["mean"], T, np.arange(T),
                                     pcast=A.PCAST_FP4, v_hat=vh)
    assert np.all(o == 2.75)


def test_equal_logits_give_the_mean_of_decoded_v():
    # all p equal 2688 -> block scale 448, code 6.0 -> decoded P = 2688 for every key
    d = np.zeros((3, 100))
    P = N.pcast_fp4(d)
    assert np.all(P == 2688.0)
    rng = np.random.default_rng(52)
    T = 256
    v = round_to_bf16(rng.standard_normal((T, 128)) * 3)
    out = N.prep_v_head_fp4(v, None, vsmooth=False)
    vh = N.vhat_fp4(out["v4"], out["sf"], out["sc"], out["mean"], T)
    zq = np.zeros((T, 128))
    qc, sq = prep.quantize_qk_head(zq)
    kc, sk = prep.quantize_qk_head(round_to_bf16(rng.standard_normal((T, 128))))
    o, _ = A.emulated_attention_head(qc, sq, kc, sk, None, None, out["mean"], T, np.arange(0, T, 9),
                                     pcast=A.PCAST_FP4, v_hat=vh)
    assert np.array_equal(o, np.broadcast_to(round_to_bf16(vh.mean(axis=0)), o.shape))


def test_p_blocks_follow_their_own_maximum():
    # a block far below the row maximum still gets a fine scale of its own
    d = np.full((1, 32), -np.inf)
    d[0, 0] = 0.0                                  # block 0: p = 2688
    d[0, 16:32] = np.log(np.linspace(1e-3, 2e-3, 16))   # block 1: p in [2.7, 5.4]
    P = N.pcast_fp4(d)
    assert P[0, 0] == 2688.0
    rel = np.abs(P[0, 16:] - 2688 * np.exp(d[0, 16:])) / (2688 * np.exp(d[0, 16:]))
    assert np.max(rel) <= 0.26                     # E2M1 half-step bound (1/4 of the top-binade value)
    assert np.all(P[0, 1:16] == 0)                 # -inf logits give 0


@pytest.mark.parametrize("vsmooth", [False, True])
def test_fp4_emulation_is_close_to_exact_attention(vsmooth):
    rng = np.random.default_rng(53)
    T = 1024
    q = round_to_bf16(rng.standard_normal((T, 128)))
    k = round_to_bf16(rng.standard_normal((T, 128)))
    v = round_to_bf16(rng.standard_normal((T, 128)) + 2)
    qc, sq = prep.quantize_qk_head(q)
    kc, sk = prep.quantize_qk_head(k)
    out = N.prep_v_head_fp4(v, None, vsmooth=vsmooth)
    vh = N.vhat_fp4(out["v4"], out["sf"], out["sc"], out["mean"], T)
    rows = np.arange(0, T, 4)
    o, _ = A.emulated_attention_head(qc, sq, kc, sk, None, None, out["mean"], T, rows,
                                     pcast=A.PCAST_FP4, v_hat=vh)
    ref = A.exact_attention_rows(q, k, v, rows)
    cos = np.sum(o * ref) / np.linalg.norm(o) / np.linalg.norm(ref)
    assert cos > 0.99
    if vsmooth:     # V-Smooth removes the +2 offset: the 4-bit residual grid is finer
        plain = N.prep_v_head_fp4(v, None, vsmooth=False)
        e_s = np.linalg.norm(vh - v)
        e_p = np.linalg.norm(N.vhat_fp4(plain["v4"], plain["sf"], plain["sc"], plain["mean"], T) - v)
        assert e_s < e_p

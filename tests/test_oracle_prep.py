"""Pins of the oracle's stage-1 prep (Q/K block quantisation, V-Smooth).

Checked against exact rational arithmetic (Python fractions), torch's
bf16 conversion, the special cases the method has, and the E4M3 error bound.
"""
from fractions import Fraction

import numpy as np
import torch

from oracle import bf16 as obf
from oracle import e4m3
from oracle import prep


def _bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _exact_bf16(q: Fraction) -> float:
    """Brute force: nearest bf16 value to a rational by scanning its neighbourhood."""
    f = abs(float(q))
    t = torch.tensor([f], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
    cands = []
    for b in range(max(t - 3, 0), min(t + 4, 0x7F80)):
        v = Fraction(obf.bf16_from_bits(np.array([b], dtype=np.uint16))[0])
        cands.append((abs(v - abs(q)), b & 1, v))
    cands.sort(key=lambda c: (c[0], c[1]))
    v = float(cands[0][2])
    return -v if q < 0 else v


def test_round_to_bf16_matches_exact_rounding():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(3000) * 10.0 ** rng.uniform(-8, 8, 3000)
    got = obf.round_to_bf16(x)
    for xi, gi in zip(x[:600], got[:600]):
        assert gi == _exact_bf16(Fraction(float(xi)))
    # values exactly representable in fp32: torch's float32 -> bf16 RNE agrees
    xf = x.astype(np.float32)
    ref = torch.from_numpy(xf).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(obf.round_to_bf16(xf.astype(np.float64)), ref)


def test_block_mean_is_exactly_rounded():
    rng = np.random.default_rng(5)
    for T in (128, 200, 77, 1):
        v = obf.bf16_from_bits(_bits(rng.standard_normal((T, 128)) * 10.0 ** rng.uniform(-3, 3, (T, 1))))
        v[0, :8] = [1e30, -1e30, 1e-30, 3e-20, 7.0, 1e25, -2e-25, 0.0]   # wide spans force exact fallbacks
        v = obf.bf16_from_bits(_bits(v))
        mu = prep.block_means(v)
        for j in range(mu.shape[0]):
            blk = v[j * 128:(j + 1) * 128]
            for c in (0, 1, 2, 3, 4, 5, 6, 7, 50, 127):
                q = sum(Fraction(float(t)) for t in blk[:, c]) / blk.shape[0]
                assert mu[j, c] == _exact_bf16(q), (T, j, c)


def test_block_mean_of_subnormal_values_is_a_bf16_value():
    """Blocks of bf16 subnormals (multiples of 2^-133): the mean of a full
    block and of a ragged one (77 rows, a rational quotient) is the nearest
    bf16 value, on the subnormal grid."""
    rng = np.random.default_rng(8)
    for T in (128, 77):
        v = rng.integers(-127, 128, size=(T, 16)).astype(np.float64) * 2.0 ** -133
        v[:, 0] = 2.0 ** -133                       # constant: mean exact
        v[:, 1] = np.where(np.arange(T) % 2, 3.0, -1.0) * 2.0 ** -133
        vp = np.zeros((T, 128))
        vp[:, :16] = v
        mu = prep.block_means(vp)
        for c in range(16):
            q = sum(Fraction(float(t)) for t in vp[:, c]) / T
            want = _exact_bf16(q)
            assert mu[0, c] == want, (T, c, mu[0, c], want)
            assert (Fraction(float(mu[0, c])) / Fraction(2) ** -133).denominator == 1
        assert mu[0, 0] == 2.0 ** -133


def test_qk_block_scale_and_codes():
    rng = np.random.default_rng(6)
    x = obf.bf16_from_bits(_bits(rng.standard_normal((200, 128)) * 3))
    codes, s = prep.quantize_qk_head(x)
    assert s.shape == (4,)
    for j in range(4):
        blk = x[j * 64:(j + 1) * 64]
        a = np.float32(np.abs(blk).max())
        assert s[j] == np.float32(a / np.float32(448))
        # the block maximum maps to +-448
        i, c = np.unravel_index(np.abs(blk).argmax(), blk.shape)
        assert codes[j * 64 + i, c] & 0x7F == 0x7E
        # dequantised error within half an E4M3 step (relative 2^-4 for normals)
        deq = e4m3.decode(codes[j * 64:(j + 1) * 64]) * s[j]
        scaled = np.abs(blk) * (448.0 / a)
        tol = np.array([[e4m3.quantum_at(max(t, 2 ** -10)) / 2 for t in row] for row in scaled]) * (a / 448.0)
        assert np.all(np.abs(deq - blk) <= tol * (1 + 1e-6) + 1e-30)


def test_qk_special_blocks():
    x = np.zeros((130, 128))
    x[64:128] = 2.5                              # identical magnitude -> all codes 448
    x[64:128, ::2] = -2.5
    x[128:] = obf.bf16_from_bits(_bits(np.linspace(-1, 1, 256).reshape(2, 128)))
    codes, s = prep.quantize_qk_head(x)
    assert s[0] == 0 and np.all(codes[:64] == 0)                     # zero block -> scale 0
    assert np.all((codes[64:128] & 0x7F) == 0x7E)
    assert np.all(codes[64:128, ::2] == 0xFE) and np.all(codes[64:128, 1::2] == 0x7E)
    assert s[2] == np.float32(np.float32(1.0) / np.float32(448))      # ragged tail block (2 rows)


def test_blocks_are_independent():
    rng = np.random.default_rng(7)
    x = obf.bf16_from_bits(_bits(rng.standard_normal((256, 128))))
    c0, s0 = prep.quantize_qk_head(x)
    y = x.copy()
    y[100, 5] = 1000.0
    c1, s1 = prep.quantize_qk_head(y)
    assert np.array_equal(c0[:64], c1[:64]) and np.array_equal(c0[128:], c1[128:])
    assert s1[1] != s0[1]


def test_v_constant_is_removed_by_the_mean():
    T = 300
    v = np.full((T, 128), 1.5)
    r = prep.prep_v_head(v, None, vsmooth=True)
    assert np.all(r["mean"] == 1.5)
    assert np.all(r["amax"] == 0) and np.all(r["sv"] == 0) and np.all(r["vq"] == 0)
    r0 = prep.prep_v_head(v, None, vsmooth=False)                   # no V-Smooth: plain channel quant
    assert np.all(r0["mean"] == 0) and np.all(r0["vq"][:, :T] == 0x7E) and np.all(r0["vq"][:, T:] == 0)


def test_v_permutation_and_layout():
    rng = np.random.default_rng(8)
    T = 333
    v = obf.bf16_from_bits(_bits(rng.standard_normal((T, 128)) + 4 * rng.standard_normal((1, 128))))
    perm = rng.permutation(T)
    a = prep.prep_v_head(v, perm, vsmooth=True)
    b = prep.prep_v_head(v[perm], None, vsmooth=True)
    for key in ("mean", "vq", "sv"):
        assert np.array_equal(a[key], b[key])
    assert a["vq"].shape == (128, 384) and np.all(a["vq"][:, T:] == 0)
    # residual scale is the channel max of |V' - mu| / 448 and the residual reconstructs V'
    # within half the largest E4M3 step (32 at the top binade) in scaled units
    resid = v[perm] - np.repeat(a["mean"], 128, axis=0)[:T]
    assert np.allclose(a["amax"], np.abs(resid).max(axis=0), rtol=1e-6)
    recon = e4m3.decode(a["vq"][:, :T]).T * a["sv"][None, :] + np.repeat(a["mean"], 128, axis=0)[:T]
    assert np.all(np.abs(recon - v[perm]) <= a["amax"][None, :] / 448 * 16 * 1.0001 + 1e-6 * np.abs(v[perm]))


def test_v_smooth_energy_removed_grows_with_cluster_order():
    # VC-Attention news article, section 2: the fraction of V energy the block
    # means remove is small in the original token order and grows once tokens
    # are sorted by cluster (8 % -> 36 % on the page's data)
    rng = np.random.default_rng(9)
    T = 2048
    cid = rng.integers(0, 16, T)
    centres = 4 * rng.standard_normal((16, 128))
    v = obf.bf16_from_bits(_bits(centres[cid] + 0.5 * rng.standard_normal((T, 128))))
    energy = np.sum(v ** 2)
    sorted_ = prep.prep_v_head(v, np.argsort(cid, kind="stable"), vsmooth=True)
    orig = prep.prep_v_head(v, None, vsmooth=True)
    removed_sorted = 1 - np.sum(sorted_["resid"].astype(np.float64) ** 2) / energy
    removed_orig = 1 - np.sum(orig["resid"].astype(np.float64) ** 2) / energy
    assert removed_sorted > 2 * removed_orig
    assert removed_sorted > 0.5

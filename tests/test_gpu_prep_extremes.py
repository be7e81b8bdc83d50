"""Prep bit-exactness on V blocks of special and extreme magnitudes.

The kernel computes a V-Smooth block mean (VC-Attention news article,
section 2 "V-Smooth": the mean of each 128-row block, kept as a 16-bit vector)
from an exact fixed-point sum and rounds it once to bf16, by one of two routes:
a full block whose values all lie inside the sum's window is an integer times
a power of two, converted without fp64; a ragged block, a block with values
below the window, or a mean outside the normal fp32 range goes through an fp64
quotient.  These cases reach every branch of both routes and compare the codes,
scales and block means with the oracle bit for bit:

* spans of 36 binades inside one block (inside the 37-binade window);
* sums that cancel exactly (mean zero), constant blocks, all-zero blocks;
* blocks of bf16 subnormals (means below the normal range: the fp64 route);
* blocks near the top of the bf16 range;
* a ragged last block of 77 rows (the fp64 route);
* the same with a random token permutation, which mixes the kinds of one head.
"""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import Workload
from tests import parity as P

pytestmark = pytest.mark.gpu

T = 8 * 128 + 77          # eight full blocks and a ragged one
H = 3


def _blk(j):
    return slice(128 * j, min(T, 128 * (j + 1)))


def _v_extremes(seed):
    g = np.random.default_rng(seed)
    v = g.standard_normal((T, H, 128))
    # head 0: wide spans inside the window, exact cancellation, constants, zeros
    v[_blk(1), 0] *= np.exp2(g.integers(-30, 7, size=(128, 128)))
    x = g.standard_normal((64, 128))
    v[_blk(2), 0] = np.concatenate([x, -x])
    v[_blk(3), 0] = g.standard_normal(128)[None, :]
    v[_blk(4), 0] = 0.0
    v[_blk(8), 0] *= np.exp2(g.integers(-20, 1, size=(77, 128)))
    # head 1: bf16 subnormals (multiples of 2^-133 below 2^-126)
    v[_blk(1), 1] = g.integers(-127, 128, size=(128, 128)) * 2.0 ** -133
    v[_blk(5), 1] = g.integers(-3, 4, size=(128, 128)) * 2.0 ** -133
    v[_blk(8), 1] = g.integers(-127, 128, size=(77, 128)) * 2.0 ** -133
    # head 2: near the top of the bf16 range
    v[_blk(1), 2] = np.clip(g.standard_normal((128, 128)), -3, 3) * 2.0 ** 124
    v[_blk(6), 2] *= 2.0 ** 100
    return v


def _workload(seed, perm):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((1, T, H, 128), generator=g).to(torch.bfloat16).cuda()
    k = torch.randn((1, T, H, 128), generator=g).to(torch.bfloat16).cuda()
    v = torch.from_numpy(_v_extremes(seed)[None]).float().to(torch.bfloat16).cuda()
    p = None
    if perm:
        p = torch.stack([torch.randperm(T, generator=g) for _ in range(H)]).to(torch.int32)[None].cuda()
    return Workload("extremes", 1, T, H, q, k, v, perm=p, vsmooth=True)


@pytest.mark.parametrize("perm", [False, True])
def test_block_means_and_codes_on_extreme_blocks(perm):
    w = _workload(31, perm)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    torch.cuda.synchronize()
    for h in range(H):
        if perm and h > 0:
            # a permutation mixes subnormal and huge values of one head into
            # blocks spanning more than the window, where the kernel's mean is
            # documented as close, not exact
            continue
        ref = P.oracle_prep_head(w, 0, h)
        P.assert_prep_bitexact(pp, ref, 0, h)
    if not perm:
        gm = pp.v_mean[0].float().cpu().numpy()
        assert np.all(gm[0, 2] == 0.0) and np.all(gm[0, 4] == 0.0)          # cancelling and zero blocks
        assert np.all((gm[1, 1] == 0.0) | (np.abs(gm[1, 1]) < 2.0 ** -126))  # subnormal means
        assert np.abs(gm[1, 1]).max() > 0.0
        assert np.abs(gm[2, 1]).max() > 2.0 ** 110

"""The seeded input recipes (bit_attention_video_e4m3_gb300/workloads.py): the
structure each workload is stated to have, checked against independent
counts (CPU only)."""
import math

import numpy as np
import torch

from bit_attention_video_e4m3_gb300.workloads import make_workload, sta_tile_lists


def _pairs_1d(n, half):
    # ordered pairs (u, v) in 0..n-1 with |u - v| <= half, counted directly
    return sum(1 for u in range(n) for v in range(n) if abs(u - v) <= half)


def test_sta_tile_lists_structure_and_density():
    grid, tile, window = (18, 48, 80), (6, 8, 8), (3, 5, 5)
    rp, cl = sta_tile_lists(grid, tile, window)
    dims = [grid[i] // tile[i] for i in range(3)]
    n3 = dims[0] * dims[1] * dims[2]
    sub = tile[0] * tile[1] * tile[2] // 128
    n = n3 * sub
    assert len(rp) == n + 1 and rp[0] == 0
    rows = [cl[rp[r]:rp[r + 1]] for r in range(n)]
    for r in rows:
        assert np.all(np.diff(r) > 0) and r.min() >= 0 and r.max() < n
    # the three 128-token tiles of one 3-D tile share its list
    for t3 in range(n3):
        for s in range(1, sub):
            assert np.array_equal(rows[t3 * sub], rows[t3 * sub + s])
    # the L-inf window is symmetric: query tile a keeps key tile b iff b keeps a
    kept = np.zeros((n, n), dtype=bool)
    for r in range(n):
        kept[r, rows[r]] = True
    assert np.array_equal(kept, kept.T)
    # the window factorises over the three axes, so the kept fraction is the
    # product of the 1-D pair counts: 22.8 % for this grid
    pairs = 1
    for d, w in zip(dims, window):
        pairs *= _pairs_1d(d, w // 2)
    assert rp[-1] == pairs * sub * sub
    assert abs(rp[-1] / n ** 2 - 0.2281) < 1e-4
    # an interior 3-D tile keeps the full 3 x 5 x 5 window
    assert max(len(r) for r in rows) == window[0] * window[1] * window[2] * sub


def test_workloads_are_reproducible_from_their_seed():
    a = make_workload("tiny", T=300, H=2)
    b = make_workload("tiny", T=300, H=2)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        assert torch.equal(x, y)
    c = make_workload("tiny", T=300, H=2, seed=5)
    assert not torch.equal(a.q, c.q)
    assert a.q.dtype == torch.bfloat16 and tuple(a.q.shape) == (1, 300, 2, 128)


def test_wan21_offset_channels():
    w = make_workload("wan21", T=2048, H=3)
    chans = w.extra["offset_channels"]
    assert len(chans) == 4 and len(set(chans)) == 4
    q = w.q.float()
    # the offset channels carry a constant per (head, channel) on top of N(0,1):
    # their token means sit far from 0 for most, the other channels' near 0
    means = q.mean(dim=1)[0]                      # [H, 128]
    other = [c for c in range(128) if c not in chans]
    assert means[:, other].abs().max() < 0.2
    assert (means[:, chans].abs() > 0.2).float().mean() > 0.5


def test_wan22_permutation_and_outliers():
    T, H = 2000, 2
    w = make_workload("wan22", T=T, H=H)
    v = w.v.float()[0]                            # [T, H, 128]
    for h in range(H):
        perm = w.perm[0, h].long()
        assert torch.equal(torch.sort(perm).values, torch.arange(T))
        norms = v[:, h].norm(dim=1)
        # 0.5 % of the rows are scaled by 20; the rest stay within a few
        # centre norms (4 sqrt(128) ~ 45)
        assert int((norms > 300).sum()) == round(0.005 * T)
        # the permutation groups rows of one cluster: neighbours in permuted
        # order are much closer than random pairs (outliers left out)
        vp = v[perm, h]
        keep = (norms[perm] < 300)
        d_next = (vp[1:] - vp[:-1]).norm(dim=1)[keep[1:] & keep[:-1]]
        d_rand = (vp - vp[torch.randperm(T)]).norm(dim=1)[keep]
        assert d_next.median() < 0.5 * d_rand.median()


def test_pcollapse_sink_logits():
    delta = 7.0
    w = make_workload("pcollapse", T=512, H=2, delta=delta)
    q, k = w.q.float()[0], w.k.float()[0]
    # channel 127 alone: q = 4 everywhere, k = delta*sqrt(128)/4 on the 4 sinks
    # and 0 elsewhere, so its logit contribution at scale 1/sqrt(128) is delta
    # on the sinks (up to the bf16 rounding of k) and 0 on every other key
    contrib = q[:, 0, 127][:, None] * k[:, 0, 127][None, :] / math.sqrt(128.0)
    assert torch.all(contrib[:, 4:] == 0)
    assert torch.allclose(contrib[:, :4], torch.full_like(contrib[:, :4], delta), rtol=2 ** -8)

"""GPU parity with two batch entries.

Every kernel addresses (batch, head) pairs: the tensor maps carry a batch
dimension, and the scales, block means, channel maxima, permutations and
sequence statistics are stored per (b, h).  Each case here gives the two
entries different data (different seeds, permutations and channel offsets)
and checks every (b, h) against the oracle: prep codes, scales and means bit
for bit, outputs within the rel-L2 tolerance overall and per row.
"""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import Workload, make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu


def _batched(T, H, seeds, offsets=False):
    """B = len(seeds) tiny-recipe entries stacked along the batch axis, each
    head with its own random permutation; with ``offsets`` every entry's K and
    V get their own per-channel offsets (so that sequence statistics differ
    between entries)."""
    parts = [make_workload("tiny", device="cuda", T=T, H=H, seed=s) for s in seeds]
    q = torch.cat([w.q for w in parts]).contiguous()
    k = torch.cat([w.k for w in parts]).contiguous()
    v = torch.cat([w.v for w in parts]).contiguous()
    B = len(seeds)
    if offsets:
        g = torch.Generator(device="cpu").manual_seed(sum(seeds))
        k = (k.float() + 3 * torch.randn(B, 1, H, 128, generator=g).cuda()).to(torch.bfloat16)
        v = (v.float() + 2 * torch.randn(B, 1, H, 128, generator=g).cuda()).to(torch.bfloat16)
    g = torch.Generator(device="cuda")
    g.manual_seed(seeds[0] * 1000 + T)
    perm = torch.stack([torch.stack([torch.randperm(T, generator=g, device="cuda") for _ in range(H)])
                        for _ in range(B)]).to(torch.int32).contiguous()
    return Workload("tiny", B, T, H, q, k, v, perm=perm, vsmooth=True)


def _sparse_lists(w, rows_l):
    w.row_ptr = torch.from_numpy(np.cumsum([0] + [len(r) for r in rows_l]).astype(np.int32)).cuda()
    w.col = torch.from_numpy(np.array(sum(rows_l, []), dtype=np.int32)).cuda()


def _check_all(w, pp, out, smooth=0, v_bias=False, n_splits=1):
    rows = np.arange(w.T)
    for b in range(w.B):
        for h in range(w.H):
            ref = P.oracle_prep_head(w, b, h, smooth=smooth, v_bias=v_bias)
            P.assert_prep_bitexact(pp, ref, b, h)
            o_ref = P.oracle_attention(w, ref, rows, n_splits=n_splits)
            got = P.gpu_rows(out, b, h, rows)
            assert P.rel_l2(got, o_ref) <= P.REL_L2_TOL, (b, h, P.rel_l2(got, o_ref))
            assert P.row_rel_l2_max(got, o_ref) <= P.ROW_REL_L2_TOL, (b, h, P.row_rel_l2_max(got, o_ref))


@pytest.mark.parametrize("pcast", [fa.PCAST_EXP2_CVT, fa.PCAST_EXPCAST])
@pytest.mark.parametrize("reverse", [False, True])
def test_two_entries_dense(pcast, reverse):
    w = _batched(333, 3, [71, 72])
    w.pcast, w.reverse = pcast, reverse
    pp, out, status = P.run_gpu(w)
    assert status == 0
    _check_all(w, pp, out)
    # the entries hold different data: their outputs must differ
    assert not torch.equal(out[0], out[1])


def test_two_entries_sparse_split():
    w = _batched(1000, 2, [73, 74])
    w.pcast = fa.PCAST_EXPCAST
    _sparse_lists(w, [[0, 1, 2, 3, 4, 5, 6, 7], [], [3], [1, 6], [0, 2, 4, 6, 7], [5], [2, 3], [7, 0, 3]])
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    for n_splits in (1, 3):
        ws = torch.empty(fa.fwd_split_workspace_bytes(w.B, w.T, w.H, n_splits), dtype=torch.uint8, device="cuda")
        out = fa.fwd(pp, row_ptr=w.row_ptr, col=w.col, pcast=w.pcast, S=w.S, beta=w.beta, vsmooth=True,
                     workspace=ws, n_splits=n_splits)
        assert fa.check_status(ws) == 0
        _check_all(w, pp, out, n_splits=n_splits)
        assert torch.all(out[:, 128:256] == 0)               # query tile 1 keeps no key tile


def test_two_entries_smoothing_and_bias():
    w = _batched(333, 2, [75, 76], offsets=True)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, smooth=2, v_bias=True)
    ws = torch.empty(fa.fwd_workspace_bytes(w.B, w.T, w.H), dtype=torch.uint8, device="cuda")
    out = fa.fwd(pp, pcast=w.pcast, S=w.S, beta=w.beta, vsmooth=True, workspace=ws)
    assert fa.check_status(ws) == 0
    _check_all(w, pp, out, smooth=2, v_bias=True)
    for b in range(w.B):
        for h in range(w.H):
            ref = P.oracle_prep_head(w, b, h, smooth=2, v_bias=True)
            off = pp.v_offset[b, h].cpu().numpy().astype(np.float64)
            tol = 1e-5 * (np.abs(ref["v_offset"]) + 1.0)
            assert np.all(np.abs(off - ref["v_offset"]) <= tol), (b, h)


def test_two_entries_fp4_pv():
    from oracle import attention as OA
    from oracle import nvfp4 as ON
    w = _batched(1000, 2, [77, 78])
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, v_format=1)
    ws = torch.empty(fa.fwd_workspace_bytes(w.B, w.T, w.H), dtype=torch.uint8, device="cuda")
    out = fa.fwd(pp, pcast=fa.PCAST_EXP2_CVT, vsmooth=True, workspace=ws)
    assert fa.check_status(ws) == 0
    rows = np.arange(w.T)
    for b in range(w.B):
        for h in range(w.H):
            ref8 = P.oracle_prep_head(w, b, h)
            _, _, v, perm = P.head_arrays(w, b, h)
            fp4 = ON.prep_v_head_fp4(v, perm, True)
            vh = ON.vhat_fp4(fp4["v4"], fp4["sf"], fp4["sc"], fp4["mean"], w.T)
            o_ref, _ = OA.emulated_attention_head(ref8["qc"], ref8["sq"], ref8["kc"], ref8["sk"], None, None,
                                                  fp4["mean"], w.T, rows, pcast=OA.PCAST_FP4, v_hat=vh)
            got = P.gpu_rows(out, b, h, rows)
            assert P.rel_l2(got, o_ref) <= P.REL_L2_TOL, (b, h, P.rel_l2(got, o_ref))

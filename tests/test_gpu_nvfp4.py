"""GPU parity of the 4-bit (NVFP4) V path against the oracle: the E2M1
conversion code by code (midpoints, saturation, signed zero), the NVFP4 V
residual (codes, UE4M3 block scales, channel scales) bit for bit, and the
4-bit PV attention within the rel-L2 tolerance."""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload
from oracle import nvfp4 as ON
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_e2m1_encode_matches_the_oracle():
    vals = [0.0, -0.0, 1e-30, -1e-30, 6.0, 6.5, 1e30, -7.0]
    for v in ON.E2M1_VALUES:
        vals += [v, -v]
    for m in (ON.E2M1_VALUES[:-1] + ON.E2M1_VALUES[1:]) / 2:
        mf = np.float32(m)
        vals += [mf, -mf, np.nextafter(mf, np.float32(0)), np.nextafter(mf, np.float32(9)),
                 -np.nextafter(mf, np.float32(0)), -np.nextafter(mf, np.float32(9))]
    rng = np.random.default_rng(60)
    dense = np.concatenate([np.array(vals, dtype=np.float32),
                            rng.uniform(-8, 8, 200000).astype(np.float32),
                            (rng.standard_normal(100000) * 0.3).astype(np.float32)])
    got = fa.e2m1_encode(torch.from_numpy(dense).cuda()).cpu().numpy()
    ref = ON.e2m1_encode(dense)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, [(float(dense[i]), int(got[i]), int(ref[i])) for i in bad[:8]]


def _unpack(pp, b, h, T):
    v4 = pp.v4[b, h].cpu().numpy()                               # [128, Tpad/2]
    codes = np.empty((128, v4.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = v4 & 0xF
    codes[:, 1::2] = v4 >> 4
    raw = pp.v4_sf[b, h].cpu().numpy()                           # [nV, 1024]
    nV = raw.shape[0]
    sf = np.empty((128, nV * 8), dtype=np.uint8)
    for kk in range(2):
        for l in range(32):
            for jj in range(4):
                for bb in range(4):
                    sf[32 * jj + l, (4 * kk + bb)::8] = raw[:, kk * 512 + l * 16 + jj * 4 + bb]
    return codes, sf, pp.v_scale[b, h].cpu().numpy()


@pytest.mark.parametrize("name,T,H,vsmooth,smooth", [
    ("tiny", 1024, 2, True, 0),
    ("tiny", 300, 2, True, 0),            # ragged: a 12-token last scale block
    ("wan22", 1500, 2, True, 0),          # permuted, clustered V with x20 outlier rows
    ("wan22", 777, 1, False, 0),
    ("tiny", 500, 2, True, 2),            # sequence-mean smoothing of K and V first
])
def test_nvfp4_v_prep_is_bit_exact(name, T, H, vsmooth, smooth):
    w = make_workload(name, device="cuda", T=T, H=H, seed=61)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=vsmooth, smooth=smooth, v_format=1)
    for h in range(H):
        ref8 = P.oracle_prep_head(w, 0, h, vsmooth=vsmooth, smooth=smooth)
        _, _, v, perm = P.head_arrays(w, 0, h)
        from oracle import smooth as OS
        vbar = OS.seq_mean_f32(v) if smooth == 2 else None
        ref = ON.prep_v_head_fp4(v, perm, vsmooth, vbar=vbar)
        codes, sf, sc = _unpack(pp, 0, h, T)
        assert np.array_equal(sc, ref["sc"]), np.flatnonzero(sc != ref["sc"])[:5]
        assert np.array_equal(sf, ref["sf"]), np.argwhere(sf != ref["sf"])[:5]
        assert np.array_equal(codes, ref["v4"]), np.argwhere(codes != ref["v4"])[:5]
        # Q/K stay E4M3 and the block means are unchanged
        assert np.array_equal(pp.q8[0, :, h].cpu().numpy(), ref8["qc"])
        assert np.array_equal(pp.k8[0, :, h].cpu().numpy(), ref8["kc"])


def _oracle_fp4(w, h, rows, vsmooth, reverse=False, n_splits=1, smooth=0):
    from oracle import attention as OA
    from oracle import smooth as OS
    ref8 = P.oracle_prep_head(w, 0, h, vsmooth=vsmooth, smooth=smooth)
    _, _, v, perm = P.head_arrays(w, 0, h)
    vbar = OS.seq_mean_f32(v) if smooth == 2 else None
    fp4 = ON.prep_v_head_fp4(v, perm, vsmooth, vbar=vbar)
    vh = ON.vhat_fp4(fp4["v4"], fp4["sf"], fp4["sc"], fp4["mean"], w.T)
    rp = None if w.row_ptr is None else w.row_ptr.cpu().numpy()
    cl = None if w.col is None else w.col.cpu().numpy()
    out, _ = OA.emulated_attention_head(ref8["qc"], ref8["sq"], ref8["kc"], ref8["sk"], None, None,
                                        fp4["mean"], w.T, rows, pcast=OA.PCAST_FP4, reverse=reverse,
                                        row_ptr=rp, col=cl, n_splits=n_splits, v_hat=vh,
                                        v_offset=None if vbar is None else vbar)
    return out


def _fwd4(w, pp, vsmooth, reverse=False, n_splits=1):
    ws = torch.empty(fa.fwd_split_workspace_bytes(w.B, w.T, w.H, n_splits), dtype=torch.uint8, device="cuda")
    out = fa.fwd(pp, row_ptr=w.row_ptr, col=w.col, reverse=reverse, pcast=fa.PCAST_EXP2_CVT,
                 vsmooth=vsmooth, workspace=ws, n_splits=n_splits)
    assert fa.check_status(ws) == 0
    return out


@pytest.mark.parametrize("name,T,H,vsmooth,reverse,n_splits", [
    ("tiny", 1024, 2, True, False, 1),
    ("tiny", 1000, 2, False, False, 1),     # ragged last key tile
    ("tiny", 1000, 2, True, True, 1),
    ("wan22", 1500, 2, True, False, 1),     # permuted clustered V with x20 outliers
    ("tiny", 1024, 2, True, False, 3),      # split-KV parts merged by log-sum-exp
])
def test_fp4_attention_parity(name, T, H, vsmooth, reverse, n_splits):
    w = make_workload(name, device="cuda", T=T, H=H, seed=62)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=vsmooth, v_format=1)
    out = _fwd4(w, pp, vsmooth, reverse, n_splits)
    for h in range(H):
        rows = np.arange(T)
        ref = _oracle_fp4(w, h, rows, vsmooth, reverse, n_splits)
        got = P.gpu_rows(out, 0, h, rows)
        assert P.rel_l2(got, ref) <= P.REL_L2_TOL, (h, P.rel_l2(got, ref))


def test_fp4_attention_sparse_and_smoothing():
    w = make_workload("tiny", device="cuda", T=1024, H=2, seed=63)
    rows_l = [[0, 1, 2, 3, 4, 5, 6, 7], [], [3], [1, 6], [0, 2, 4, 6, 7], [5], [2, 3], [7, 0, 3]]
    w.row_ptr = torch.from_numpy(np.cumsum([0] + [len(r) for r in rows_l]).astype(np.int32)).cuda()
    w.col = torch.from_numpy(np.array(sum(rows_l, []), dtype=np.int32)).cuda()
    w.v = (w.v.float() * 2 + 3).to(torch.bfloat16)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, smooth=2, v_format=1)
    out = _fwd4(w, pp, True)
    for h in range(w.H):
        rows = np.arange(w.T)
        ref = _oracle_fp4(w, h, rows, True, smooth=2)
        got = P.gpu_rows(out, 0, h, rows)
        assert P.rel_l2(got, ref) <= P.REL_L2_TOL
    assert torch.all(out[0, 128:256].float() == 0)


def test_fp4_constant_v_is_exact():
    w = make_workload("tiny", device="cuda", T=700, H=1, seed=64)
    w.v = torch.full_like(w.v, -1.625)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, v_format=1)
    assert torch.all(_fwd4(w, pp, True).float() == -1.625)


@pytest.mark.parametrize("T", [1, 17, 63, 129, 300])
def test_fp4_attention_ragged_lengths(T):
    w = make_workload("tiny", device="cuda", T=T, H=2, seed=100 + T)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, v_format=1)
    out = _fwd4(w, pp, True)
    for h in range(w.H):
        rows = np.arange(T)
        ref = _oracle_fp4(w, h, rows, True)
        assert P.rel_l2(P.gpu_rows(out, 0, h, rows), ref) <= P.REL_L2_TOL

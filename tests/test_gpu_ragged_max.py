"""Row maximum on ragged key tiles (GPU, through the C ABI).

On a full tile the kernel takes the row maximum from the score loads
themselves (the reducing TMEM load returns the largest of the columns it
reads); the key columns of a ragged last tile past T hold the scores of zero
keys, i.e. 0.  Here every real score lies far below zero (about -45 in natural
units), so a maximum that let the padded columns in would put every
probability of the row 2^-65 below the static scale and cast it to code 0.
Checked against the oracle for both P casts, both visiting orders (reverse
order visits the ragged tile first), with V-Smooth, 4-bit PV and split-KV.
"""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload
from oracle import attention as OA
from oracle import nvfp4 as ON
from tests import parity as P

pytestmark = pytest.mark.gpu


def _far_below_zero(T, H, seed):
    w = make_workload("tiny", device="cuda", T=T, H=H, seed=seed)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    shape = w.q.shape
    w.q = torch.full(shape, 2.0, device="cuda").to(w.q.dtype)
    w.k = (-2.0 + 0.25 * torch.randn(shape, generator=g, device="cuda")).to(w.k.dtype)
    return w


def _assert_close_to_exact(out, w, ref, rows):
    got = P.gpu_rows(out, 0, 0, rows)
    assert np.abs(got).max() > 0.0
    assert P.cosine(got, P.exact_attention(w, ref, rows)) > 0.95


@pytest.mark.parametrize("T", [100, 300])
@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("pcast", [fa.PCAST_EXP2_CVT, fa.PCAST_EXPCAST])
@pytest.mark.parametrize("vsmooth", [False, True])
def test_padded_keys_stay_out_of_the_row_max(T, reverse, pcast, vsmooth):
    w = _far_below_zero(T, 2, seed=T + 7)
    w.reverse, w.pcast, w.vsmooth = reverse, pcast, vsmooth
    pp, out, status = P.run_gpu(w)
    assert status == 0
    rows = np.arange(T)
    for h in range(w.H):
        ref = P.oracle_prep_head(w, 0, h, vsmooth=vsmooth)
        o_ref = P.oracle_attention(w, ref, rows)
        assert P.rel_l2(P.gpu_rows(out, 0, h, rows), o_ref) <= P.REL_L2_TOL
    _assert_close_to_exact(out, w, P.oracle_prep_head(w, 0, 0, vsmooth=vsmooth), rows)


@pytest.mark.parametrize("T", [100, 300])
def test_padded_keys_stay_out_of_the_row_max_split(T):
    w = _far_below_zero(T, 2, seed=T + 8)
    w.vsmooth = False
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=False)
    ws = torch.empty(fa.fwd_split_workspace_bytes(w.B, w.T, w.H, 2), dtype=torch.uint8, device="cuda")
    out = fa.fwd(pp, pcast=fa.PCAST_EXP2_CVT, vsmooth=False, workspace=ws, n_splits=2)
    assert fa.check_status(ws) == 0
    rows = np.arange(T)
    for h in range(w.H):
        ref = P.oracle_prep_head(w, 0, h, vsmooth=False)
        o_ref = P.oracle_attention(w, ref, rows, pcast=fa.PCAST_EXP2_CVT, n_splits=2)
        assert P.rel_l2(P.gpu_rows(out, 0, h, rows), o_ref) <= P.REL_L2_TOL


@pytest.mark.parametrize("T", [100, 300])
@pytest.mark.parametrize("reverse", [False, True])
def test_padded_keys_stay_out_of_the_block_maxima_fp4(T, reverse):
    # 4-bit PV: the block maxima of the 16-key scale blocks come from the same
    # reducing loads; a ragged tile recomputes them over its valid keys
    w = _far_below_zero(T, 1, seed=T + 9)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, v_format=1)
    ws = torch.empty(fa.fwd_split_workspace_bytes(w.B, w.T, w.H, 1), dtype=torch.uint8, device="cuda")
    out = fa.fwd(pp, reverse=reverse, pcast=fa.PCAST_EXP2_CVT, vsmooth=True, workspace=ws, n_splits=1)
    assert fa.check_status(ws) == 0
    ref8 = P.oracle_prep_head(w, 0, 0, vsmooth=True)
    _, _, v, perm = P.head_arrays(w, 0, 0)
    fp4 = ON.prep_v_head_fp4(v, perm, True)
    vh = ON.vhat_fp4(fp4["v4"], fp4["sf"], fp4["sc"], fp4["mean"], w.T)
    rows = np.arange(T)
    o_ref, _ = OA.emulated_attention_head(ref8["qc"], ref8["sq"], ref8["kc"], ref8["sk"], None, None,
                                          fp4["mean"], w.T, rows, pcast=OA.PCAST_FP4, reverse=reverse,
                                          v_hat=vh)
    assert P.rel_l2(P.gpu_rows(out, 0, 0, rows), o_ref) <= P.REL_L2_TOL
    _assert_close_to_exact(out, w, ref8, rows)

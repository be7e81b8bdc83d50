"""GPU parity of split-KV (fp8attn_fwd_split) against the oracle's split
emulation: every part of a query tile's visiting order runs its own online
softmax and the parts are merged by a log-sum-exp reduction.  Outputs are
checked within the rel-L2 tolerance, on dense, reversed, ragged and sparse
lists (with empty parts), with V-Smooth and with the smoothing offset;
n_splits = 1 must reproduce fp8attn_fwd bit for bit."""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu


def _fwd(w, pp, n_splits, **kw):
    ws = torch.empty(fa.fwd_split_workspace_bytes(w.B, w.T, w.H, max(n_splits, 1)), dtype=torch.uint8,
                     device="cuda")
    args = dict(row_ptr=w.row_ptr, col=w.col, reverse=w.reverse, pcast=w.pcast, S=w.S, beta=w.beta,
                vsmooth=w.vsmooth)
    args.update(kw)
    out = fa.fwd(pp, workspace=ws, n_splits=n_splits, **args)
    assert fa.check_status(ws) == 0
    return out


def _check(w, pp, out, n_splits, reverse=None, pcast=None, smooth=0, v_bias=False, rows=None):
    for h in range(w.H):
        ref = P.oracle_prep_head(w, 0, h, smooth=smooth, v_bias=v_bias)
        rr = np.arange(w.T) if rows is None else rows
        o_ref = P.oracle_attention(w, ref, rr, reverse=reverse, pcast=pcast, n_splits=n_splits)
        got = P.gpu_rows(out, 0, h, rr)
        assert P.rel_l2(got, o_ref) <= P.REL_L2_TOL, (h, P.rel_l2(got, o_ref))


@pytest.mark.parametrize("n_splits", [2, 3, 8])
@pytest.mark.parametrize("pcast", [fa.PCAST_EXP2_CVT, fa.PCAST_EXPCAST])
@pytest.mark.parametrize("reverse", [False, True])
def test_split_parity_dense(n_splits, pcast, reverse):
    w = make_workload("tiny", device="cuda", T=1000, H=2, seed=21)      # 8 key tiles, ragged tail
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    out = _fwd(w, pp, n_splits, pcast=pcast, reverse=reverse)
    _check(w, pp, out, n_splits, reverse=reverse, pcast=pcast)


def test_split_one_is_the_plain_kernel():
    import ctypes
    w = make_workload("tiny", device="cuda", T=777, H=2, seed=22)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    a = _fwd(w, pp, 1)                                          # fp8attn_fwd
    b = torch.empty_like(a)
    ws = torch.empty(fa.fwd_split_workspace_bytes(w.B, w.T, w.H, 1), dtype=torch.uint8, device="cuda")
    st = pp._struct()
    code = fa.lib().fp8attn_fwd_split(ctypes.byref(st), w.B, w.T, w.H, 128, None, None, 0, int(w.pcast),
                                      float(w.S), float(w.beta), 0.0, 1, 1, b.data_ptr(),
                                      ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert code == 0 and fa.check_status(ws) == 0
    assert torch.equal(a, b)


def test_split_parity_sparse_with_empty_parts():
    # a CSR list with empty rows and rows shorter than the number of parts
    w = make_workload("tiny", device="cuda", T=1024, H=2, seed=23)
    rows = [[0, 1, 2, 3, 4, 5, 6, 7], [], [3], [1, 6], [0, 2, 4, 6, 7], [5], [], [7, 0, 3]]
    rp = np.cumsum([0] + [len(r) for r in rows]).astype(np.int32)
    col = np.array(sum(rows, []), dtype=np.int32)
    w.row_ptr = torch.from_numpy(rp).cuda()
    w.col = torch.from_numpy(col).cuda()
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    for n_splits in (2, 4):
        out = _fwd(w, pp, n_splits)
        _check(w, pp, out, n_splits)
        o = out.float()
        assert torch.all(o[0, 128:256] == 0) and torch.all(o[0, 768:896] == 0)     # empty lists


def test_split_with_smoothing_offset_and_constant_v():
    w = make_workload("tiny", device="cuda", T=900, H=2, seed=24)
    w.v = (w.v.float() * 2 + 3).to(torch.bfloat16)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, smooth=2, v_bias=True)
    out = _fwd(w, pp, 3)
    _check(w, pp, out, 3, smooth=2, v_bias=True)
    c = make_workload("tiny", device="cuda", T=700, H=1, seed=25)
    c.v = torch.full_like(c.v, -1.75)
    ppc = fa.prep(c.q, c.k, c.v, perm=c.perm, vsmooth=True)
    assert torch.all(_fwd(c, ppc, 4).float() == -1.75)


def test_auto_split_on_a_small_problem_and_closeness_to_unsplit():
    w = make_workload("tiny", device="cuda", T=4096, H=1, seed=26)     # 32 query tiles < 152 SMs
    n = fa.auto_splits(w.B, w.T, w.H)
    assert n > 1
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    a = _fwd(w, pp, 1).float()
    b = _fwd(w, pp, n).float()
    assert torch.equal(b, fa.fwd(pp, vsmooth=True, n_splits=0).float())      # auto = the same split
    rows = P.sample_rows(w.T, 384, seed=3)
    _check(w, pp, b, n, rows=rows)
    # each part casts P against its own running max: the split is as close to
    # exact attention as the unsplit kernel (the oracle's split pin states the same)
    ref = P.oracle_prep_head(w, 0, 0)
    exact = P.exact_attention(w, ref, rows)
    e_split = np.linalg.norm(P.gpu_rows(b.to(torch.bfloat16), 0, 0, rows) - exact)
    e_plain = np.linalg.norm(P.gpu_rows(a.to(torch.bfloat16), 0, 0, rows) - exact)
    assert e_split <= 1.5 * e_plain


@pytest.mark.parametrize("T,n_splits", [(1, 3), (129, 2), (200, 4), (63, 2)])
def test_split_ragged_and_empty_parts(T, n_splits):
    # fewer key tiles than parts leaves parts empty; they must not disturb the merge
    w = make_workload("tiny", device="cuda", T=T, H=2, seed=200 + T)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    out = _fwd(w, pp, n_splits)
    _check(w, pp, out, n_splits)

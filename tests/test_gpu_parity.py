"""GPU parity of the CUDA path against the oracle on small and ragged inputs.

Prep: codes, scales and block means bit-exact.  Attention: rel-L2 <= 5e-3
against the oracle's emulated-quantisation output on every row; cosine
against exact fp64 attention is printed.  All calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload, sta_tile_lists
from tests import parity as P

pytestmark = pytest.mark.gpu


def _check(w, heads=None, rows=None, **kw):
    pp, out, status = P.run_gpu(w, **kw)
    assert status == 0, fa._lib.Fp8AttnError(status, "device status")
    heads = heads if heads is not None else [(0, h) for h in range(w.H)]
    worst = 0.0
    for b, h in heads:
        ref = P.oracle_prep_head(w, b, h, vsmooth=kw.get("vsmooth"))
        P.assert_prep_bitexact(pp, ref, b, h)
        r = np.arange(w.T) if rows is None else rows
        o_ref = P.oracle_attention(w, ref, r, **{k: v for k, v in kw.items() if k != "vsmooth"})
        got = P.gpu_rows(out, b, h, r)
        rel = P.rel_l2(got, o_ref)
        worst = max(worst, rel)
        assert rel <= P.REL_L2_TOL, (b, h, rel)
        row_worst = P.row_rel_l2_max(got, o_ref)
        assert row_worst <= P.ROW_REL_L2_TOL, (b, h, "worst row", row_worst)
    return pp, out, worst


@pytest.mark.parametrize("pcast", [fa.PCAST_EXP2_CVT, fa.PCAST_EXPCAST])
@pytest.mark.parametrize("vsmooth", [False, True])
@pytest.mark.parametrize("reverse", [False, True])
def test_tiny(pcast, vsmooth, reverse):
    w = make_workload("tiny", device="cuda", vsmooth=vsmooth)
    w.pcast = pcast
    w.reverse = reverse
    _, out, worst = _check(w)
    ref = P.oracle_prep_head(w, 0, 0)
    rows = np.arange(0, w.T, 4)
    cos = P.cosine(P.gpu_rows(out, 0, 0, rows), P.exact_attention(w, ref, rows))
    print(f"tiny pcast={pcast} vsmooth={vsmooth} reverse={reverse}: rel-L2 {worst:.2e}, cos(exact) {cos:.5f}")
    assert cos > 0.99


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 129, 200, 333, 1000])
def test_ragged_lengths(T):
    w = make_workload("tiny", device="cuda", T=T, H=3, seed=T)
    g = torch.Generator(device="cuda")
    g.manual_seed(T)
    w.perm = torch.stack([torch.randperm(T, generator=g, device="cuda") for _ in range(3)]).to(torch.int32)[None].contiguous()
    w.pcast = fa.PCAST_EXPCAST if T % 2 else fa.PCAST_EXP2_CVT
    _check(w)


def test_sparse_sliding_tile_small():
    # grid 12 x 16 x 32 of 6x8x8 tiles -> 2 x 2 x 4 = 16 tiles of 384 tokens
    grid = (12, 16, 32)
    w = make_workload("sta", device="cuda", H=2, grid=grid)
    _, _, worst = _check(w)
    rp, cl = sta_tile_lists(grid=grid, window=(3, 3, 3))
    w.row_ptr = torch.from_numpy(rp).cuda()
    w.col = torch.from_numpy(cl).cuda()
    _check(w)
    w.reverse = True
    _check(w)


@pytest.mark.parametrize("reverse", [False, True])
def test_vsmooth_expcast_with_ragged_sparse_lists(reverse):
    """V-Smooth (permuted V) and ExpCast on per-query-tile key-tile lists of
    every length from empty to full, unsorted: the mean-term pipeline sees
    every tile count (its final step depends on the count's parity) and
    empty tiles give zero rows."""
    w = make_workload("tiny", device="cuda", T=1100, H=2, seed=41, vsmooth=True)
    n = -(-w.T // 128)                                   # 9 query and key tiles, the last ragged
    g = np.random.default_rng(41)
    lengths = [0, 1, 2, 3, 4, 5, 9, 6, 7]
    lists = [g.permutation(n)[:k] for k in lengths[:n]]
    rp = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int32)
    cl = np.concatenate(lists).astype(np.int32)
    w.row_ptr = torch.from_numpy(rp).cuda()
    w.col = torch.from_numpy(cl).cuda()
    gt = torch.Generator(device="cuda")
    gt.manual_seed(41)
    w.perm = torch.stack([torch.randperm(w.T, generator=gt, device="cuda") for _ in range(w.H)]).to(torch.int32)[None].contiguous()
    w.pcast = fa.PCAST_EXPCAST
    w.reverse = reverse
    _, out, _ = _check(w)
    assert torch.all(out[0, :128] == 0)                 # the empty list


def test_sparse_full_list_is_bit_identical_to_dense():
    w = make_workload("tiny", device="cuda", T=700, H=2)
    n = -(-w.T // 128)
    rp = torch.arange(0, n * n + 1, n, dtype=torch.int32, device="cuda")
    cl = torch.arange(n, dtype=torch.int32, device="cuda").repeat(n)
    for rev in (False, True):
        _, dense, _ = P.run_gpu(w, reverse=rev, row_ptr=None, col=None)
        _, sparse, _ = P.run_gpu(w, reverse=rev, row_ptr=rp, col=cl)
        assert torch.equal(dense, sparse)


def test_empty_and_unsorted_tile_lists():
    w = make_workload("tiny", device="cuda", T=512, H=2)
    rp = torch.tensor([0, 0, 2, 3, 6], dtype=torch.int32, device="cuda")
    cl = torch.tensor([3, 1, 2, 0, 3, 1], dtype=torch.int32, device="cuda")
    pp, out, status = P.run_gpu(w, row_ptr=rp, col=cl)
    assert status == 0
    assert torch.all(out[0, :128] == 0)
    for h in range(w.H):
        ref = P.oracle_prep_head(w, 0, h)
        rows = np.arange(w.T)
        o_ref = P.oracle_attention(w, ref, rows, row_ptr=rp, col=cl)
        assert P.rel_l2(P.gpu_rows(out, 0, h, rows), o_ref) <= P.REL_L2_TOL


def test_bad_tile_index_is_reported_not_faulted():
    w = make_workload("tiny", device="cuda", T=256, H=1)
    rp = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    cl = torch.tensor([0, 5], dtype=torch.int32, device="cuda")      # 5 >= nV = 2
    _, _, status = P.run_gpu(w, row_ptr=rp, col=cl)
    assert status == 6      # FP8ATTN_ERR_BAD_TILE_LIST


@pytest.mark.parametrize("pcast", [fa.PCAST_EXP2_CVT, fa.PCAST_EXPCAST])
def test_constant_v_is_preserved_exactly(pcast):
    w = make_workload("tiny", device="cuda", T=333, H=2)
    w.v = torch.full_like(w.v, -2.375)
    w.pcast = pcast
    _, out, status = P.run_gpu(w, vsmooth=True)
    assert status == 0
    assert torch.all(out == -2.375)


def test_zero_queries_give_the_mean_of_dequantised_v():
    w = make_workload("tiny", device="cuda", T=200, H=2)
    w.q = torch.zeros_like(w.q)
    _check(w)


def test_invalid_arguments_are_rejected():
    w = make_workload("tiny", device="cuda", T=128, H=1)
    pp = fa.prep(w.q, w.k, w.v)
    with pytest.raises(fa.Fp8AttnError) as e:
        fa.fwd(pp, S=0.5)
    assert e.value.code == 1
    with pytest.raises(fa.Fp8AttnError) as e:
        fa.fwd(pp, S=256.0, pcast=7)
    assert e.value.code == 1
    with pytest.raises(fa.Fp8AttnError) as e:
        fa.fwd(pp, workspace=torch.empty(8, dtype=torch.uint8, device="cuda"))
    assert e.value.code == 5


# ExpCast at the top of the code range: the row maximum's code is
# rne(8 log2 S + 56 + beta), which reaches 127 (E4M3's NaN pattern) for S = 448
# and beta >= 0.04, so the cast must clamp at 126 (VC-Attention news article,
# section 3; the clamp keeps every P code finite).
@pytest.mark.parametrize("S,beta", [(448.0, 0.05), (448.0, 0.3), (448.0, 0.45), (440.0, 0.45),
                                    (1.0, 0.45), (256.0, 0.45), (448.0, -0.49)])
@pytest.mark.parametrize("T", [1024, 333])
def test_expcast_code_range_and_top_clamp(S, beta, T):
    w = make_workload("tiny", device="cuda", T=T, H=2, seed=int(S) + T)
    w.pcast = fa.PCAST_EXPCAST
    w.S = S
    w.beta = beta
    _, out, _ = _check(w)
    assert torch.isfinite(out.float()).all()


def test_permutation_entry_out_of_range_is_reported_not_faulted():
    w = make_workload("tiny", device="cuda", T=300, H=2)
    perm = w.perm.clone()
    perm[0, 1, 17] = w.T + 5          # outside [0, T)
    perm[0, 0, 3] = -1
    pp = fa.prep(w.q, w.k, w.v, perm=perm, vsmooth=True,
                 workspace=(ws := torch.empty(fa.prep_workspace_bytes(w.B, w.T, w.H), dtype=torch.uint8,
                                              device="cuda")))
    assert fa.check_status(ws) == 7       # FP8ATTN_ERR_BAD_PERMUTATION
    assert fa.check_status(ws) == 0       # read and cleared
    # the same call with the valid permutation reports nothing and matches the oracle
    fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, out=pp, workspace=ws)
    assert fa.check_status(ws) == 0
    for h in range(w.H):
        P.assert_prep_bitexact(pp, P.oracle_prep_head(w, 0, h), 0, h)


def test_plain_prep_and_fwd_entry_points_through_ctypes():
    """fp8attn_prep and fp8attn_fwd themselves (the two calls of the boundary),
    called directly with valid data, against the oracle."""
    import ctypes
    L = fa.lib()
    w = make_workload("tiny", device="cuda", T=700, H=3, seed=11)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    w.perm = torch.stack([torch.randperm(w.T, generator=g, device="cuda") for _ in range(w.H)]
                         ).to(torch.int32)[None].contiguous()
    w.pcast = fa.PCAST_EXPCAST
    pp = fa.Prepped.empty(w.B, w.T, w.H, "cuda")
    st = pp._struct()
    nws = int(L.fp8attn_workspace_size(w.B, w.T, w.H, 128))
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    code = L.fp8attn_prep(w.q.data_ptr(), w.k.data_ptr(), w.v.data_ptr(), w.B, w.T, w.H, 128,
                          w.perm.data_ptr(), 1, ctypes.byref(st), ws.data_ptr(), nws, stream)
    assert code == 0
    out = torch.empty_like(w.q)
    code = L.fp8attn_fwd(ctypes.byref(st), w.B, w.T, w.H, 128, None, None, 0, fa.PCAST_EXPCAST,
                         ctypes.c_float(256.0), ctypes.c_float(-0.35), ctypes.c_float(0.0), 1,
                         out.data_ptr(), ws.data_ptr(), nws, stream)
    assert code == 0
    assert L.fp8attn_check_status(ws.data_ptr(), stream) == 0
    rows = np.arange(w.T)
    for h in range(w.H):
        ref = P.oracle_prep_head(w, 0, h)
        P.assert_prep_bitexact(pp, ref, 0, h)
        o_ref = P.oracle_attention(w, ref, rows)
        got = P.gpu_rows(out, 0, h, rows)
        assert P.rel_l2(got, o_ref) <= P.REL_L2_TOL
        assert P.row_rel_l2_max(got, o_ref) <= P.ROW_REL_L2_TOL


# V-Smooth adds its block-mean terms in batches of four key tiles, read from a
# ring of eight TMEM row-sum columns well after their PV products; the last
# batch follows the last tile.  Tile counts of every residue mod 4, odd and even
# (the last tile belongs to either softmax group), each run four times: the
# output must repeat bit for bit (a batch read too early would not) and match
# the oracle.
@pytest.mark.parametrize("T", [777, 1024, 1290, 4173, 4352, 4480, 4600])
@pytest.mark.parametrize("pcast", [fa.PCAST_EXP2_CVT, fa.PCAST_EXPCAST])
def test_vsmooth_batches_repeat_bit_for_bit(T, pcast):
    w = make_workload("tiny", device="cuda", T=T, H=2, seed=T + 7)
    w.pcast = pcast
    pp, out, _ = _check(w, rows=P.sample_rows(w.T, 384, seed=1))
    for _ in range(3):
        again = fa.fwd(pp, pcast=pcast, S=w.S, beta=w.beta, vsmooth=True)
        assert torch.equal(out, again)

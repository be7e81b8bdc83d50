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

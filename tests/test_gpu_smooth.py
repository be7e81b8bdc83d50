"""GPU parity of sequence-mean smoothing (fp8attn_prep_smooth) against the
oracle: codes, scales and block means bit-exact (they can only match if the
GPU's fp32 sequence means equal the oracle's exactly rounded ones), the output
offset within fp32 summation noise, outputs within the rel-L2 tolerance."""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu


def _run(w, smooth, v_bias):
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=w.vsmooth, smooth=smooth, v_bias=v_bias)
    ws = torch.empty(fa.fwd_workspace_bytes(w.B, w.T, w.H), dtype=torch.uint8, device="cuda")
    out = fa.fwd(pp, pcast=w.pcast, S=w.S, beta=w.beta, vsmooth=w.vsmooth, workspace=ws)
    assert fa.check_status(ws) == 0
    return pp, out


@pytest.mark.parametrize("smooth,v_bias", [(1, False), (2, False), (0, True), (2, True)])
@pytest.mark.parametrize("vsmooth", [False, True])
def test_smoothing_parity(smooth, v_bias, vsmooth):
    w = make_workload("tiny", device="cuda", T=333, H=2, seed=7, vsmooth=vsmooth)
    # channel offsets make the K centring matter
    g = torch.Generator(device="cpu").manual_seed(5)
    w.k = (w.k.float() + 3 * torch.randn(1, 1, w.H, 128, generator=g).cuda()).to(torch.bfloat16)
    w.v = (w.v.float() + 2 * torch.randn(1, 1, w.H, 128, generator=g).cuda()).to(torch.bfloat16)
    pp, out = _run(w, smooth, v_bias)
    for h in range(w.H):
        ref = P.oracle_prep_head(w, 0, h, smooth=smooth, v_bias=v_bias)
        P.assert_prep_bitexact(pp, ref, 0, h)
        if ref["v_offset"] is None:          # K-only smoothing adds nothing to the output
            assert pp.v_offset is None
        else:
            off = pp.v_offset[0, h].cpu().numpy().astype(np.float64)
            tol = 1e-5 * (np.abs(ref["v_offset"]) + 1.0)
            assert np.all(np.abs(off - ref["v_offset"]) <= tol), np.max(np.abs(off - ref["v_offset"]))
        rows = np.arange(w.T)
        got = P.gpu_rows(out, 0, h, rows)
        o_ref = P.oracle_attention(w, ref, rows)
        assert P.rel_l2(got, o_ref) <= P.REL_L2_TOL


def test_plain_prep_writes_a_zero_offset():
    w = make_workload("tiny", device="cuda", T=200, H=1, seed=3)
    out = fa.Prepped.empty(w.B, w.T, w.H, "cuda", with_offset=True)
    out.v_offset.fill_(7.0)
    fa.prep(w.q, w.k, w.v, vsmooth=True, out=out)
    assert torch.all(out.v_offset == 0)


def test_uniform_weights_restore_the_mean_of_v():
    w = make_workload("tiny", device="cuda", T=500, H=2, seed=9, vsmooth=True)
    w.q = torch.zeros_like(w.q)
    w.v = (w.v.float() * 2 + 5).to(torch.bfloat16)
    _, out = _run(w, 2, True)
    mean_v = w.v.float().mean(dim=1, keepdim=True)
    err = (out.float() - mean_v).abs()
    assert torch.all(err <= mean_v.abs() * 2.0 ** -8 + 1e-4), err.max()


def test_k_smoothing_improves_accuracy_on_channel_offsets():
    w = make_workload("wan21", device="cuda", T=2048, H=2, seed=13)
    rows = np.arange(0, w.T, 4)
    errs = []
    for smooth in (0, 1):
        _, out = _run(w, smooth, False)
        e = []
        for h in range(w.H):
            ref = P.oracle_prep_head(w, 0, h)
            ex = P.exact_attention(w, ref, rows)
            e.append(P.rel_l2(P.gpu_rows(out, 0, h, rows), ex))
        errs.append(np.mean(e))
    print("rel-L2 vs exact attention, no smoothing / K smoothing:", errs)
    assert errs[1] < 0.95 * errs[0]

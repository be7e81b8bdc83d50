"""GPU parity of the last-wave split (fp8attn_fwd_tail_split).

The query tiles of the whole waves run exactly as in fp8attn_fwd and must be
bit-identical.  Each last-wave query tile runs in parts that first take the
row maxima of the key tiles before their range, so they cast the unsplit P
codes: their rows may differ from fp8attn_fwd only by the fp32 rounding order
of the log-sum-exp merge (at most one bf16 step), and they must match the
oracle's unsplit emulation within the rel-L2 tolerance.  The SM count passed
in only shapes the plan; any value is correct on any device.
"""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu


def _workload(T, H, seed, vsmooth):
    w = make_workload("tiny", device="cuda", T=T, H=H, seed=seed, vsmooth=vsmooth)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    w.perm = torch.stack([torch.randperm(T, generator=g, device="cuda") for _ in range(H)]).to(torch.int32)[None].contiguous()
    return w


def _run(w, pp, pcast, reverse, vsmooth, num_sms):
    ws0 = torch.empty(fa.fwd_workspace_bytes(w.B, w.T, w.H), dtype=torch.uint8, device="cuda")
    a = fa.fwd(pp, pcast=pcast, S=w.S, beta=w.beta, reverse=reverse, vsmooth=vsmooth, workspace=ws0)
    assert fa.check_status(ws0) == 0
    ws1 = torch.empty(fa.fwd_tail_workspace_bytes(w.B, w.T, w.H, num_sms), dtype=torch.uint8, device="cuda")
    b = fa.fwd(pp, pcast=pcast, S=w.S, beta=w.beta, reverse=reverse, vsmooth=vsmooth, workspace=ws1,
               tail_split=True, num_sms=num_sms)
    assert fa.check_status(ws1) == 0
    return a, b


def _tail_tiles(w, num_sms):
    """(b, h, qt) of the last-wave query tiles, by linear CTA index qt + nQt (h + H b)."""
    parts, nt, lo = fa.tail_plan(w.B, w.T, w.H, num_sms)
    nqt = -(-w.T // 128)
    total = w.B * w.H * nqt
    return parts, [(c // nqt // w.H, (c // nqt) % w.H, c % nqt) for c in range(total - nt, total)]


@pytest.mark.parametrize("T,H,num_sms", [(1000, 3, 10), (4000, 2, 20)])
@pytest.mark.parametrize("pcast", [fa.PCAST_EXP2_CVT, fa.PCAST_EXPCAST])
@pytest.mark.parametrize("vsmooth", [False, True])
@pytest.mark.parametrize("reverse", [False, True])
def test_tail_split_keeps_the_unsplit_codes(T, H, num_sms, pcast, vsmooth, reverse):
    w = _workload(T, H, T + num_sms, vsmooth)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=vsmooth)
    parts, tail = _tail_tiles(w, num_sms)
    assert parts >= 2 and tail
    a, b = _run(w, pp, pcast, reverse, vsmooth, num_sms)
    in_tail = torch.zeros((w.B, w.H, -(-w.T // 128)), dtype=torch.bool)
    for bb, h, qt in tail:
        in_tail[bb, h, qt] = True
    for bb in range(w.B):
        for h in range(w.H):
            for qt in range(-(-w.T // 128)):
                r0, r1 = qt * 128, min(w.T, qt * 128 + 128)
                x, y = a[bb, r0:r1, h].float(), b[bb, r0:r1, h].float()
                if not in_tail[bb, h, qt]:
                    assert torch.equal(x, y), (bb, h, qt)          # the whole waves: the plain kernel
                    continue
                # the same P codes: only the merge's fp32 rounding order differs (one
                # bf16 step, or a few fp32 roundings of the tile's scale near zero)
                step = torch.maximum(x.abs(), y.abs()) * 2.0 ** -7 + 1e-5 * x.abs().max()
                assert torch.all((x - y).abs() <= step), (bb, h, qt, float((x - y).abs().max()))
                assert float((x == y).float().mean()) >= 0.99, (bb, h, qt)
    # the last-wave rows against the oracle's unsplit emulation
    for h in sorted({h for _, h, _ in tail}):
        rows = np.concatenate([np.arange(qt * 128, min(w.T, qt * 128 + 128)) for bb, hh, qt in tail if hh == h])
        ref = P.oracle_prep_head(w, 0, h, vsmooth=vsmooth)
        o_ref = P.oracle_attention(w, ref, rows, reverse=reverse, pcast=pcast)
        got = P.gpu_rows(b, 0, h, rows)
        assert P.rel_l2(got, o_ref) <= P.REL_L2_TOL, (h, P.rel_l2(got, o_ref))
        assert P.row_rel_l2_max(got, o_ref) <= P.ROW_REL_L2_TOL


def test_without_a_plan_the_call_is_the_plain_kernel():
    w = _workload(1000, 3, 5, True)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    for sms in (24, 8, 200):                    # whole waves; whole waves; a single wave
        assert fa.tail_plan(1, 1000, 3, sms)[0] == 1
        a, b = _run(w, pp, fa.PCAST_EXPCAST, False, True, sms)
        assert torch.equal(a, b)


def test_tail_split_with_the_smoothing_offset_and_two_entries():
    # two batch entries, sequence-mean smoothing of K and V with the bias
    # correction (an output offset the merge adds), on a plan of 3 parts
    parts_w = [make_workload("tiny", device="cuda", T=2000, H=2, seed=s) for s in (81, 82)]
    q = torch.cat([x.q for x in parts_w]).contiguous()
    k = torch.cat([x.k for x in parts_w]).contiguous()
    v = (torch.cat([x.v for x in parts_w]).float() * 2 + 1).to(torch.bfloat16).contiguous()
    pp = fa.prep(q, k, v, vsmooth=True, smooth=2, v_bias=True)
    plan = fa.tail_plan(2, 2000, 2, 18)                     # 64 query tiles on 18 SMs: 3 waves + 10
    assert plan[0] == 1                                      # 10 > 18 / 2: kept whole
    plan = fa.tail_plan(2, 2000, 2, 20)                      # 3 waves + 4: 3 parts
    assert plan[0] >= 2
    ws0 = torch.empty(fa.fwd_workspace_bytes(2, 2000, 2), dtype=torch.uint8, device="cuda")
    a = fa.fwd(pp, pcast=fa.PCAST_EXP2_CVT, vsmooth=True, workspace=ws0)
    ws1 = torch.empty(fa.fwd_tail_workspace_bytes(2, 2000, 2, 20), dtype=torch.uint8, device="cuda")
    b = fa.fwd(pp, pcast=fa.PCAST_EXP2_CVT, vsmooth=True, workspace=ws1, tail_split=True, num_sms=20)
    assert fa.check_status(ws0) == 0 and fa.check_status(ws1) == 0
    x, y = a.float(), b.float()
    step = torch.maximum(x.abs(), y.abs()) * 2.0 ** -7 + 1e-5 * x.abs().amax(dim=(1, 3), keepdim=True)
    assert torch.all((x - y).abs() <= step)
    assert float((x == y).float().mean()) >= 0.995
    assert not torch.equal(a[0], a[1])


def test_tail_split_rejects_tile_lists_and_fp4():
    w = _workload(1000, 1, 9, True)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    rp = torch.tensor([0, 1, 2, 3, 4, 5, 6, 7, 8], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        fa.fwd(pp, row_ptr=rp, col=rp[:8].clone(), tail_split=True, num_sms=10)
    pp4 = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True, v_format=1)
    with pytest.raises(ValueError):
        fa.fwd(pp4, tail_split=True, num_sms=10)

"""fp8attn_prep_noalloc — the prep call for callers that cannot allocate device
memory (it keeps its scratch in a fixed array inside the library) — must give
exactly what fp8attn_prep gives, and what the oracle gives.  Called through the
C ABI twice in a row, with different inputs, so that scratch left over from the
first call would show."""
import ctypes

import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300._lib import Prepped, _Prepped
from bit_attention_video_e4m3_gb300.workloads import make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu

FIELDS = ("q8", "k8", "v8", "q_scale", "k_scale", "v_scale", "v_mean")
ERR_WORKSPACE = 5
MAX_BH = 2048


def _entry():
    f = fa.lib().fp8attn_prep_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, i, i, i, i, vp, i, ctypes.POINTER(_Prepped), vp]
    f.restype = i
    return f


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else (
        t.view(torch.int32) if t.dtype == torch.float32 else t)


def _workload(seed, scale):
    w = make_workload("tiny", device="cuda", T=333, H=3, seed=seed)
    w.v = (w.v.float() * scale).to(torch.bfloat16)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    perm = torch.stack([torch.randperm(w.T, generator=g, device="cuda") for _ in range(w.H)])
    w.perm = perm.to(torch.int32)[None].contiguous()
    return w


def test_prep_noalloc_matches_prep_on_two_calls_in_a_row():
    f = _entry()
    stream = torch.cuda.current_stream().cuda_stream
    # the first call leaves large channel maxima behind; the second call has small ones
    for seed, scale in ((7, 50.0), (8, 0.5)):
        w = _workload(seed, scale)
        ref = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
        got = Prepped.empty(w.B, w.T, w.H, w.q.device)
        st = got._struct()
        code = f(w.q.data_ptr(), w.k.data_ptr(), w.v.data_ptr(), w.B, w.T, w.H, 128,
                 w.perm.data_ptr(), 1, ctypes.byref(st), stream)
        assert code == 0, fa.lib().fp8attn_status_string(code)
        torch.cuda.synchronize()
        for name in FIELDS:
            assert torch.equal(_bits(getattr(got, name)), _bits(getattr(ref, name))), name
        # and, on its own, bit-exact with the oracle's prep of every head
        for h in range(w.H):
            P.assert_prep_bitexact(got, P.oracle_prep_head(w, 0, h, vsmooth=True), 0, h)


def test_prep_noalloc_rejects_problems_beyond_its_scratch():
    f = _entry()
    w = make_workload("tiny", device="cuda", T=64, H=1)
    got = Prepped.empty(w.B, w.T, w.H, w.q.device)
    st = got._struct()
    # B*H one past the fixed capacity: refused before any work is queued
    code = f(w.q.data_ptr(), w.k.data_ptr(), w.v.data_ptr(), 1, 64, MAX_BH + 1, 128, None, 1,
             ctypes.byref(st), torch.cuda.current_stream().cuda_stream)
    assert code == ERR_WORKSPACE

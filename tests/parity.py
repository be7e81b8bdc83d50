"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare.  Test infrastructure only."""
from __future__ import annotations

import math

import numpy as np
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import bf16_bits
from oracle import attention as OA
from oracle import prep as OP
from oracle import smooth as OS
from oracle.bf16 import bf16_from_bits

REL_L2_TOL = 5e-3     # output tolerance vs the emulated oracle (stated by the method's target)


def run_gpu(w, reverse=None, pcast=None, S=None, vsmooth=None, row_ptr="w", col="w"):
    vs = w.vsmooth if vsmooth is None else vsmooth
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=vs)
    ws = torch.empty(fa.fwd_workspace_bytes(w.B, w.T, w.H), dtype=torch.uint8, device=w.q.device)
    rp = w.row_ptr if isinstance(row_ptr, str) else row_ptr
    cl = w.col if isinstance(col, str) else col
    out = fa.fwd(pp, row_ptr=rp, col=cl, reverse=w.reverse if reverse is None else reverse,
                 pcast=w.pcast if pcast is None else pcast, S=w.S if S is None else S,
                 beta=w.beta, vsmooth=vs, workspace=ws)
    status = fa.check_status(ws)
    return pp, out, status


def head_arrays(w, b, h):
    """bf16 values (fp64) of one head's Q, K, V in original order, and its permutation."""
    q = bf16_from_bits(bf16_bits(w.q[b, :, h, :]))
    k = bf16_from_bits(bf16_bits(w.k[b, :, h, :]))
    v = bf16_from_bits(bf16_bits(w.v[b, :, h, :]))
    perm = None if w.perm is None else w.perm[b, h].cpu().numpy().astype(np.int64)
    return q, k, v, perm


def oracle_prep_head(w, b, h, vsmooth=None, smooth=0, v_bias=False):
    """Oracle stage 1 of one head; with sequence-mean smoothing (smooth 1: K,
    2: K and V) and the V bias correction the result also holds the output
    offset ``v_offset`` (fp64 [128])."""
    vs = w.vsmooth if vsmooth is None else vsmooth
    q, k, v, perm = head_arrays(w, b, h)
    qc, sq = OP.quantize_qk_head(q)
    kk = OS.center(k, OS.seq_mean_f32(k)) if smooth >= 1 else k
    kc, sk = OP.quantize_qk_head(kk if perm is None else kk[perm])
    vbar = OS.seq_mean_f32(v) if smooth == 2 else None
    pv = OP.prep_v_head(v, perm, vs, vbar=vbar)
    off = None
    if smooth == 2 or v_bias:
        off = np.zeros(128) if vbar is None else vbar.astype(np.float64)
        if v_bias:
            off = off - OS.v_bias(pv["vq"], pv["sv"], pv["mean"], pv["vprime"])
    return dict(qc=qc, sq=sq, kc=kc, sk=sk, vq=pv["vq"], sv=pv["sv"], mean=pv["mean"],
                q=q, k=k, v=v, perm=perm, v_offset=off)


def assert_prep_bitexact(pp, ref, b, h):
    np.testing.assert_array_equal(pp.q8[b, :, h].cpu().numpy(), ref["qc"], err_msg="q codes")
    np.testing.assert_array_equal(pp.q_scale[b, h].cpu().numpy().view(np.uint32),
                                  ref["sq"].view(np.uint32), err_msg="q scales")
    np.testing.assert_array_equal(pp.k8[b, :, h].cpu().numpy(), ref["kc"], err_msg="k codes")
    np.testing.assert_array_equal(pp.k_scale[b, h].cpu().numpy().view(np.uint32),
                                  ref["sk"].view(np.uint32), err_msg="k scales")
    np.testing.assert_array_equal(pp.v8[b, h].cpu().numpy(), ref["vq"], err_msg="v codes")
    np.testing.assert_array_equal(pp.v_scale[b, h].cpu().numpy().view(np.uint32),
                                  ref["sv"].view(np.uint32), err_msg="v scales")
    gm = pp.v_mean[b, h].float().cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(gm, ref["mean"], err_msg="v block means")


def oracle_attention(w, ref, rows, reverse=None, pcast=None, S=None, row_ptr="w", col="w", n_splits=1):
    rp = w.row_ptr if isinstance(row_ptr, str) else row_ptr
    cl = w.col if isinstance(col, str) else col
    rp = None if rp is None else rp.cpu().numpy()
    cl = None if cl is None else cl.cpu().numpy()
    out, _ = OA.emulated_attention_head(
        ref["qc"], ref["sq"], ref["kc"], ref["sk"], ref["vq"], ref["sv"], ref["mean"], w.T, rows,
        pcast=w.pcast if pcast is None else pcast, S=w.S if S is None else S, beta=w.beta,
        reverse=w.reverse if reverse is None else reverse, row_ptr=rp, col=cl,
        v_offset=ref.get("v_offset"), n_splits=n_splits)
    return out


def exact_attention(w, ref, rows, row_ptr="w", col="w"):
    """fp64 attention from the bf16 inputs (same kept key tiles when sparse)."""
    rp = w.row_ptr if isinstance(row_ptr, str) else row_ptr
    cl = w.col if isinstance(col, str) else col
    k = ref["k"] if ref["perm"] is None else ref["k"][ref["perm"]]
    v = ref["v"] if ref["perm"] is None else ref["v"][ref["perm"]]
    mask_fn = None
    if rp is not None:
        rpn, cln = rp.cpu().numpy(), cl.cpu().numpy()
        n_t = -(-w.T // 128)

        def mask_fn(r):
            qt = r // 128
            return OA.kept_key_mask(w.T, OA.tile_list_for_qtile(qt, n_t, False, rpn, cln))
    return OA.exact_attention_rows(ref["q"], k, v, rows, key_mask_for_row=mask_fn)


def rel_l2(got, ref):
    d = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / d) if d > 0 else float(np.linalg.norm(got))


# Per-row bound: a single wrong row (wrong tile, wrong max, wrong scale) has a
# relative error of order one, which a norm over hundreds of rows can dilute
# below REL_L2_TOL; rows that merely see a few P codes rounded the other way
# stay far below this.
ROW_REL_L2_TOL = 4 * REL_L2_TOL


def row_rel_l2_max(got, ref):
    """Largest relative L2 error of any single row (rows with a zero reference
    norm count their absolute error)."""
    num = np.linalg.norm(got - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    r = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    return float(r.max()) if r.size else 0.0


def cosine(a, b):
    return float(np.sum(a * b) / (np.linalg.norm(a) * np.linalg.norm(b)))


def sample_rows(T, n=256, seed=0):
    """n query rows spread over [0, T) including the first and the ragged-tail rows."""
    rng = np.random.default_rng(seed)
    tail = list(range(max(0, T - 8), T))
    head = [0, 1, 127, 128] if T > 128 else [0]
    k = max(0, n - len(tail) - len(head))
    mid = rng.choice(T, size=min(k, T), replace=False).tolist()
    return np.unique(np.array([r for r in head + mid + tail if r < T], dtype=np.int64))


def gpu_rows(out, b, h, rows):
    return out[b, :, h, :].float().cpu().numpy().astype(np.float64)[rows]

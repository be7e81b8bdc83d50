"""ctypes binding of libfp8attn.so (argument marshalling only).

Names follow the C ABI: ``prep`` -> fp8attn_prep_smooth (fp8attn_prep when smooth == 0
and no bias correction; fp8attn_prep_ex for an NVFP4 V), ``fwd`` -> fp8attn_fwd
(fp8attn_fwd_split for split-KV, fp8attn_fwd_ex for 4-bit PV),
``check_status`` -> fp8attn_check_status, ``e4m3_encode`` -> fp8attn_e4m3_encode,
``v_cluster`` -> fp8attn_v_cluster.  Outputs and workspaces are torch
tensors on the current CUDA device; the stream is torch's current stream
unless one is passed.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

PCAST_EXP2_CVT = 0
PCAST_EXPCAST = 1
HEAD_DIM = 128

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def library_path() -> str:
    return os.path.join(_HERE, "libfp8attn.so")


class Fp8AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        name = lib().fp8attn_status_string(code).decode()
        super().__init__(f"{where}: {name} (status {code})")
        self.code = code


class _Prepped(ctypes.Structure):
    _fields_ = [("q8", ctypes.c_void_p), ("k8", ctypes.c_void_p), ("v8", ctypes.c_void_p),
                ("q_scale", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("v_mean", ctypes.c_void_p),
                ("v_offset", ctypes.c_void_p), ("v4", ctypes.c_void_p), ("v4_sf", ctypes.c_void_p)]


def lib():
    """Load libfp8attn.so (built in-tree by build.build_library)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() (nvcc, sm_103a) first")
        L = ctypes.CDLL(path)
        i, f, vp, sz = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
        L.fp8attn_workspace_size.argtypes = [i, i, i, i]
        L.fp8attn_workspace_size.restype = sz
        L.fp8attn_prep_workspace_bytes.argtypes = [i, i, i]
        L.fp8attn_prep_workspace_bytes.restype = sz
        L.fp8attn_fwd_workspace_bytes.argtypes = [i, i, i]
        L.fp8attn_fwd_workspace_bytes.restype = sz
        L.fp8attn_v_padded_T.argtypes = [i]
        L.fp8attn_v_padded_T.restype = sz
        L.fp8attn_abi_version.argtypes = []
        L.fp8attn_abi_version.restype = i
        L.fp8attn_status_string.argtypes = [i]
        L.fp8attn_status_string.restype = ctypes.c_char_p
        L.fp8attn_prep.argtypes = [vp, vp, vp, i, i, i, i, vp, i, ctypes.POINTER(_Prepped), vp, sz, vp]
        L.fp8attn_prep.restype = i
        L.fp8attn_prep_smooth.argtypes = [vp, vp, vp, i, i, i, i, vp, i, i, i,
                                          ctypes.POINTER(_Prepped), vp, sz, vp]
        L.fp8attn_prep_smooth.restype = i
        L.fp8attn_fwd.argtypes = [ctypes.POINTER(_Prepped), i, i, i, i, vp, vp, i, i, f, f, f, i,
                                  vp, vp, sz, vp]
        L.fp8attn_fwd.restype = i
        L.fp8attn_check_status.argtypes = [vp, vp]
        L.fp8attn_check_status.restype = i
        L.fp8attn_e4m3_encode.argtypes = [vp, vp, sz, vp]
        L.fp8attn_e4m3_encode.restype = i
        L.fp8attn_e2m1_encode.argtypes = [vp, vp, sz, vp]
        L.fp8attn_e2m1_encode.restype = i
        L.fp8attn_prep_ex.argtypes = [vp, vp, vp, i, i, i, i, vp, i, i, i, i,
                                      ctypes.POINTER(_Prepped), vp, sz, vp]
        L.fp8attn_prep_ex.restype = i
        L.fp8attn_fwd_split.argtypes = [ctypes.POINTER(_Prepped), i, i, i, i, vp, vp, i, i, f, f, f, i, i,
                                        vp, vp, sz, vp]
        L.fp8attn_fwd_split.restype = i
        L.fp8attn_fwd_ex.argtypes = [ctypes.POINTER(_Prepped), i, i, i, i, vp, vp, i, i, f, f, f, i, i, i,
                                     vp, vp, sz, vp]
        L.fp8attn_fwd_ex.restype = i
        L.fp8attn_fwd_split_workspace_bytes.argtypes = [i, i, i, i]
        L.fp8attn_fwd_split_workspace_bytes.restype = sz
        L.fp8attn_fwd_auto_splits.argtypes = [i, i, i, i]
        L.fp8attn_fwd_auto_splits.restype = i
        L.fp8attn_fwd_tail_split.argtypes = [ctypes.POINTER(_Prepped), i, i, i, i, i, i, f, f, f, i, i,
                                             vp, vp, sz, vp]
        L.fp8attn_fwd_tail_split.restype = i
        L.fp8attn_fwd_tail_workspace_bytes.argtypes = [i, i, i, i]
        L.fp8attn_fwd_tail_workspace_bytes.restype = sz
        L.fp8attn_fwd_tail_plan.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        L.fp8attn_fwd_tail_plan.restype = i
        L.fp8attn_selftest_wait_timeout.argtypes = [vp, ctypes.c_ulonglong, vp]
        L.fp8attn_selftest_wait_timeout.restype = i
        L.fp8attn_cluster_workspace_bytes.argtypes = [i, i, i, i]
        L.fp8attn_cluster_workspace_bytes.restype = sz
        L.fp8attn_v_cluster.argtypes = [vp, i, i, i, i, i, i, i, vp, vp, vp, sz, vp]
        L.fp8attn_v_cluster.restype = i
        _LIB = L
    return _LIB


@dataclass
class Prepped:
    """Stage-1 outputs (device tensors) of a [B, T, H, 128] problem."""
    B: int
    T: int
    H: int
    q8: torch.Tensor        # uint8 [B,T,H,128]
    k8: torch.Tensor        # uint8 [B,T,H,128] (permuted key order)
    v8: torch.Tensor        # uint8 [B,H,128,Tpad]
    q_scale: torch.Tensor   # fp32 [B,H,nQK]
    k_scale: torch.Tensor   # fp32 [B,H,nQK]
    v_scale: torch.Tensor   # fp32 [B,H,128]
    v_mean: torch.Tensor    # bf16 [B,H,nV,128]
    v_offset: torch.Tensor | None = None   # fp32 [B,H,128] added to every output row
    v4: torch.Tensor | None = None         # uint8 [B,H,128,Tpad/2] packed E2M1 (NVFP4 V)
    v4_sf: torch.Tensor | None = None      # uint8 [B,H,nV,1024] UE4M3 block scales of v4

    @staticmethod
    def empty(B: int, T: int, H: int, device, with_offset: bool = False, v_format: int = 0) -> "Prepped":
        nqk = -(-T // 64)
        nv = -(-T // 128)
        u8 = dict(dtype=torch.uint8, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        fp4 = v_format == 1
        return Prepped(B, T, H,
                       torch.empty((B, T, H, HEAD_DIM), **u8), torch.empty((B, T, H, HEAD_DIM), **u8),
                       torch.empty((0,), **u8) if fp4 else torch.empty((B, H, HEAD_DIM, nv * 128), **u8),
                       torch.empty((B, H, nqk), **f32), torch.empty((B, H, nqk), **f32),
                       torch.empty((B, H, HEAD_DIM), **f32),
                       torch.empty((B, H, nv, HEAD_DIM), dtype=torch.bfloat16, device=device),
                       torch.empty((B, H, HEAD_DIM), **f32) if with_offset else None,
                       torch.empty((B, H, HEAD_DIM, nv * 64), **u8) if fp4 else None,
                       torch.empty((B, H, nv, 1024), **u8) if fp4 else None)

    @property
    def v_format(self) -> int:
        return 1 if self.v4 is not None else 0

    def _struct(self) -> _Prepped:
        return _Prepped(self.q8.data_ptr(), self.k8.data_ptr(),
                        None if self.v4 is not None else self.v8.data_ptr(),
                        self.q_scale.data_ptr(), self.k_scale.data_ptr(), self.v_scale.data_ptr(),
                        self.v_mean.data_ptr(),
                        None if self.v_offset is None else self.v_offset.data_ptr(),
                        None if self.v4 is None else self.v4.data_ptr(),
                        None if self.v4_sf is None else self.v4_sf.data_ptr())


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_input(t: torch.Tensor, name: str, dtype):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prep_workspace_bytes(B: int, T: int, H: int) -> int:
    return int(lib().fp8attn_prep_workspace_bytes(B, T, H))


def fwd_workspace_bytes(B: int, T: int, H: int) -> int:
    return int(lib().fp8attn_fwd_workspace_bytes(B, T, H))


def prep(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, perm: torch.Tensor | None = None,
         vsmooth: bool = True, out: Prepped | None = None, workspace: torch.Tensor | None = None,
         stream=None, smooth: int = 0, v_bias: bool = False, v_format: int = 0) -> Prepped:
    """fp8attn_prep_ex: bf16 [B,T,H,128] Q, K, V (+ int32 [B,H,T] permutation) ->
    Prepped.  smooth: 0 none, 1 centre K, 2 centre K and V over the sequence;
    v_bias: compensate the measured E4M3 mean bias of V (both need the output
    offset, allocated here when ``out`` is not given); v_format: 0 E4M3 residual,
    1 NVFP4 residual (for the 4-bit PV product)."""
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check_input(t, nm, torch.bfloat16)
    B, T, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    if perm is not None:
        _check_input(perm, "perm", torch.int32)
        if tuple(perm.shape) != (B, H, T):
            raise ValueError("perm must be [B, H, T]")
    if out is None:
        out = Prepped.empty(B, T, H, q.device, with_offset=(smooth == 2 or bool(v_bias)), v_format=v_format)
    if workspace is None:
        workspace = torch.empty(prep_workspace_bytes(B, T, H), dtype=torch.uint8, device=q.device)
    st = out._struct()
    code = lib().fp8attn_prep_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, D,
                                 None if perm is None else perm.data_ptr(), int(bool(vsmooth)),
                                 int(smooth), int(bool(v_bias)), int(v_format), ctypes.byref(st),
                                 workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if code != 0:
        raise Fp8AttnError(code, "fp8attn_prep_ex")
    return out


def fwd_split_workspace_bytes(B: int, T: int, H: int, n_splits: int) -> int:
    return int(lib().fp8attn_fwd_split_workspace_bytes(B, T, H, n_splits))


def auto_splits(B: int, T: int, H: int, num_sms: int | None = None) -> int:
    """fp8attn_fwd_auto_splits on the current device's SM count (or num_sms)."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return int(lib().fp8attn_fwd_auto_splits(B, T, H, int(num_sms)))


def fwd_tail_workspace_bytes(B: int, T: int, H: int, num_sms: int) -> int:
    return int(lib().fp8attn_fwd_tail_workspace_bytes(B, T, H, num_sms))


def _num_sms(device) -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


def tail_plan(B: int, T: int, H: int, num_sms: int | None = None):
    """fp8attn_fwd_tail_plan: (parts, n_tail, part_lo) of the last-wave split on
    num_sms SMs (default: the current device's); parts 1 keeps the last wave whole."""
    if num_sms is None:
        num_sms = _num_sms(torch.cuda.current_device())
    nt = ctypes.c_int(0)
    lo = (ctypes.c_int * 5)()
    parts = int(lib().fp8attn_fwd_tail_plan(B, T, H, int(num_sms), ctypes.byref(nt), lo))
    return parts, int(nt.value), [int(lo[k]) for k in range(parts + 1)] if parts >= 2 else []


def fwd(pp: Prepped, row_ptr: torch.Tensor | None = None, col: torch.Tensor | None = None,
        reverse: bool = False, pcast: int = PCAST_EXP2_CVT, S: float = 256.0, beta: float = -0.35,
        softmax_scale: float = 0.0, vsmooth: bool = True, out: torch.Tensor | None = None,
        workspace: torch.Tensor | None = None, stream=None, n_splits: int = 1,
        tail_split: bool = False, num_sms: int | None = None) -> torch.Tensor:
    """fp8attn_fwd (n_splits == 1) / fp8attn_fwd_split / fp8attn_fwd_ex (NVFP4 V):
    prepared operands -> bf16 [B,T,H,128] output.  n_splits = 0 picks
    fp8attn_fwd_auto_splits.  A Prepped holding an NVFP4 V (prep(..., v_format=1))
    runs the 4-bit PV product.  tail_split (dense, 8-bit PV, n_splits 1):
    fp8attn_fwd_tail_split on num_sms SMs (default: the device's), the last
    wave's query tiles split with the unsplit P codes."""
    B, T, H = pp.B, pp.T, pp.H
    if tail_split:
        if row_ptr is not None or col is not None or n_splits != 1 or pp.v_format == 1:
            raise ValueError("tail_split is for dense attention with the 8-bit PV product and n_splits 1")
        if num_sms is None:
            num_sms = _num_sms(pp.q8.device)
        if out is None:
            out = torch.empty((B, T, H, HEAD_DIM), dtype=torch.bfloat16, device=pp.q8.device)
        if workspace is None:
            workspace = torch.empty(fwd_tail_workspace_bytes(B, T, H, num_sms), dtype=torch.uint8,
                                    device=pp.q8.device)
        st = pp._struct()
        code = lib().fp8attn_fwd_tail_split(ctypes.byref(st), B, T, H, HEAD_DIM, int(bool(reverse)), int(pcast),
                                            float(S), float(beta), float(softmax_scale), int(bool(vsmooth)),
                                            int(num_sms), out.data_ptr(), workspace.data_ptr(),
                                            workspace.numel(), _stream_handle(stream))
        if code != 0:
            raise Fp8AttnError(code, "fp8attn_fwd_tail_split")
        return out
    if n_splits == 0:
        n_splits = auto_splits(B, T, H)
    if (row_ptr is None) != (col is None):
        raise ValueError("row_ptr and col go together")
    if row_ptr is not None:
        _check_input(row_ptr, "row_ptr", torch.int32)
        _check_input(col, "col", torch.int32)
        if row_ptr.numel() != -(-T // 128) + 1:
            raise ValueError("row_ptr must have ceil(T/128)+1 entries")
    if out is None:
        out = torch.empty((B, T, H, HEAD_DIM), dtype=torch.bfloat16, device=pp.q8.device)
    if workspace is None:
        workspace = torch.empty(fwd_split_workspace_bytes(B, T, H, n_splits), dtype=torch.uint8,
                                device=pp.q8.device)
    st = pp._struct()
    common = (None if row_ptr is None else row_ptr.data_ptr(), None if col is None else col.data_ptr(),
              int(bool(reverse)), int(pcast), float(S), float(beta), float(softmax_scale),
              int(bool(vsmooth)))
    tail = (out.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if pp.v_format == 1:
        code = lib().fp8attn_fwd_ex(ctypes.byref(st), B, T, H, HEAD_DIM, *common, int(n_splits), 1, *tail)
        name = "fp8attn_fwd_ex"
    elif n_splits == 1:
        code = lib().fp8attn_fwd(ctypes.byref(st), B, T, H, HEAD_DIM, *common, *tail)
        name = "fp8attn_fwd"
    else:
        code = lib().fp8attn_fwd_split(ctypes.byref(st), B, T, H, HEAD_DIM, *common, int(n_splits), *tail)
        name = "fp8attn_fwd_split"
    if code != 0:
        raise Fp8AttnError(code, name)
    return out


def e4m3_encode(x: torch.Tensor, stream=None) -> torch.Tensor:
    """fp8attn_e4m3_encode: E4M3 codes (uint8, same shape) of a float32 CUDA tensor."""
    if x.dtype != torch.float32 or not x.is_cuda:
        raise ValueError("x must be a float32 CUDA tensor")
    x = x.contiguous()
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    st = lib().fp8attn_e4m3_encode(x.data_ptr(), codes.data_ptr(), x.numel(), _stream_handle(stream))
    if st != 0:
        raise Fp8AttnError(st, "fp8attn_e4m3_encode")
    return codes


def cluster_workspace_bytes(B: int, T: int, H: int, n_dims: int = 8) -> int:
    return int(lib().fp8attn_cluster_workspace_bytes(B, T, H, n_dims))


def v_cluster(v: torch.Tensor, n_clusters: int = 32, n_dims: int = 8, iters: int = 4,
              with_labels: bool = False, perm: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None):
    """fp8attn_v_cluster: bf16 [B,T,H,128] V -> int32 [B,H,T] permutation (the stable
    sort of the tokens by cluster), plus the int32 [B,H,T] cluster ids if asked."""
    _check_input(v, "v", torch.bfloat16)
    B, T, H, D = v.shape
    if perm is None:
        perm = torch.empty((B, H, T), dtype=torch.int32, device=v.device)
    labels = torch.empty((B, H, T), dtype=torch.int32, device=v.device) if with_labels else None
    if workspace is None:
        workspace = torch.empty(cluster_workspace_bytes(B, T, H, n_dims), dtype=torch.uint8,
                                device=v.device)
    code = lib().fp8attn_v_cluster(v.data_ptr(), B, T, H, D, int(n_clusters), int(n_dims), int(iters),
                                   perm.data_ptr(), None if labels is None else labels.data_ptr(),
                                   workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if code != 0:
        raise Fp8AttnError(code, "fp8attn_v_cluster")
    return (perm, labels) if with_labels else perm


def e2m1_encode(x: torch.Tensor, stream=None) -> torch.Tensor:
    """fp8attn_e2m1_encode: E2M1 codes (uint8, low nibble, same shape) of a float32 CUDA tensor."""
    if x.dtype != torch.float32 or not x.is_cuda:
        raise ValueError("x must be a float32 CUDA tensor")
    x = x.contiguous()
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    st = lib().fp8attn_e2m1_encode(x.data_ptr(), codes.data_ptr(), x.numel(), _stream_handle(stream))
    if st != 0:
        raise Fp8AttnError(st, "fp8attn_e2m1_encode")
    return codes


def selftest_wait_timeout(workspace: torch.Tensor, limit_ns: int, stream=None) -> None:
    """fp8attn_selftest_wait_timeout: a bounded wait that nothing ends (see the header)."""
    code = lib().fp8attn_selftest_wait_timeout(workspace.data_ptr(), int(limit_ns), _stream_handle(stream))
    if code != 0:
        raise Fp8AttnError(code, "fp8attn_selftest_wait_timeout")


def check_status(workspace: torch.Tensor, stream=None) -> int:
    """fp8attn_check_status: synchronise and return (and clear) a kernel status code."""
    return int(lib().fp8attn_check_status(workspace.data_ptr(), _stream_handle(stream)))

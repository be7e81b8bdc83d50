"""Block-scaled FP8 (E4M3) attention forward for video DiTs on GB300 (sm_103a).

Two stages behind a C ABI (include/fp8attn.h, libfp8attn.so):
  prep(q, k, v, perm, vsmooth)       bf16 [B,T,H,128] -> E4M3 codes + scales (+ V block means)
  fwd(prepped, ..., n_splits=1)      -> bf16 [B,T,H,128] attention output (split-KV when n_splits > 1)
  v_cluster(v)                       -> int32 [B,H,T] V-Smooth permutation (online V clustering)
This package only marshals torch tensors into the C ABI; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback:
calls fail loudly if the library is missing or the device is not sm_103.
"""
from ._lib import (PCAST_EXP2_CVT, PCAST_EXPCAST, Fp8AttnError, Prepped, check_status,
                   e2m1_encode, e4m3_encode, fwd, lib, library_path, prep, prep_workspace_bytes,
                   fwd_workspace_bytes, v_cluster, cluster_workspace_bytes, auto_splits,
                   fwd_split_workspace_bytes, selftest_wait_timeout, tail_plan, fwd_tail_workspace_bytes)

__all__ = ["prep", "fwd", "check_status", "e2m1_encode", "e4m3_encode", "Prepped", "Fp8AttnError", "PCAST_EXP2_CVT",
           "PCAST_EXPCAST", "lib", "library_path", "prep_workspace_bytes", "fwd_workspace_bytes",
           "v_cluster", "cluster_workspace_bytes", "auto_splits", "fwd_split_workspace_bytes", "selftest_wait_timeout",
           "tail_plan", "fwd_tail_workspace_bytes"]

"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8attn.h")


@pytest.fixture(scope="module")
def L():
    from bit_attention_video_e4m3_gb300.build import build_library
    build_library()
    import bit_attention_video_e4m3_gb300 as fa
    return fa.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8attn_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"fp8attn_prep", "fp8attn_fwd", "fp8attn_check_status"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_host_helpers(L):
    assert L.fp8attn_abi_version() == 7
    assert L.fp8attn_v_padded_T(1) == 128
    assert L.fp8attn_v_padded_T(32760) == 32768
    assert L.fp8attn_v_padded_T(75600) == 75648
    assert L.fp8attn_prep_workspace_bytes(1, 1000, 40) >= 40 * 128 * 4
    assert L.fp8attn_fwd_workspace_bytes(1, 1000, 40) >= 4
    L.fp8attn_workspace_size.restype = ctypes.c_size_t
    assert L.fp8attn_workspace_size(1, 1000, 40, 128) == max(L.fp8attn_prep_workspace_bytes(1, 1000, 40),
                                                             L.fp8attn_fwd_workspace_bytes(1, 1000, 40))
    assert L.fp8attn_workspace_size(1, 1000, 40, 64) == 0
    assert L.fp8attn_cluster_workspace_bytes(1, 75600, 40, 8) >= 40 * 75600 * (16 + 1)
    assert L.fp8attn_cluster_workspace_bytes(1, 100, 1, 17) == 0
    for code in range(8):
        assert L.fp8attn_status_string(code)
        assert L.fp8attn_status_string(code) != b"unknown status"
    assert L.fp8attn_status_string(7) == b"permutation entry out of range"


def test_bad_arguments_rejected_before_any_cuda_call(L):
    from bit_attention_video_e4m3_gb300._lib import _Prepped
    pp = _Prepped(16, 16, 16, 16, 16, 16, 16)
    # D != 128
    assert L.fp8attn_prep(16, 16, 16, 1, 64, 1, 64, None, 1, ctypes.byref(pp), 16, 1 << 20, None) == 1
    # null input
    assert L.fp8attn_prep(None, 16, 16, 1, 64, 1, 128, None, 1, ctypes.byref(pp), 16, 1 << 20, None) == 1
    # misaligned pointer
    assert L.fp8attn_prep(17, 16, 16, 1, 64, 1, 128, None, 1, ctypes.byref(pp), 16, 1 << 20, None) == 1
    # workspace too small
    assert L.fp8attn_prep(16, 16, 16, 1, 64, 1, 128, None, 1, ctypes.byref(pp), 16, 8, None) == 5
    # smoothing: mode out of range, bias flag out of range, missing output offset
    ws = L.fp8attn_prep_workspace_bytes(1, 64, 1)
    assert L.fp8attn_prep_smooth(16, 16, 16, 1, 64, 1, 128, None, 1, 3, 0, ctypes.byref(pp), 16, ws, None) == 1
    assert L.fp8attn_prep_smooth(16, 16, 16, 1, 64, 1, 128, None, 1, 1, 2, ctypes.byref(pp), 16, ws, None) == 1
    assert L.fp8attn_prep_smooth(16, 16, 16, 1, 64, 1, 128, None, 1, 2, 0, ctypes.byref(pp), 16, ws, None) == 1
    assert L.fp8attn_prep_smooth(16, 16, 16, 1, 64, 1, 128, None, 1, 0, 1, ctypes.byref(pp), 16, ws, None) == 1
    # fwd: S out of range, bad pcast, half a CSR
    args = dict(B=1, T=64, H=1)
    base = [ctypes.byref(pp), 1, 64, 1, 128]
    assert L.fp8attn_fwd(*base, None, None, 0, 0, ctypes.c_float(0.5), ctypes.c_float(-0.35),
                         ctypes.c_float(0), 1, 16, 16, 256, None) == 1
    assert L.fp8attn_fwd(*base, None, None, 0, 3, ctypes.c_float(256), ctypes.c_float(-0.35),
                         ctypes.c_float(0), 1, 16, 16, 256, None) == 1
    assert L.fp8attn_fwd(*base, 16, None, 0, 0, ctypes.c_float(256), ctypes.c_float(-0.35),
                         ctypes.c_float(0), 1, 16, 16, 256, None) == 1
    assert L.fp8attn_fwd(*base, None, None, 0, 0, ctypes.c_float(256), ctypes.c_float(0.7),
                         ctypes.c_float(0), 1, 16, 16, 256, None) == 1


def test_empty_and_oversized_shapes_rejected(L):
    """B, T or H of zero, more than 65535 heads, more than 32767 batches, or
    B * H * T beyond 31 bits: argument errors from prep and fwd, found before
    any CUDA call (the boundary has no zero-work path)."""
    from bit_attention_video_e4m3_gb300._lib import _Prepped
    pp = _Prepped(16, 16, 16, 16, 16, 16, 16)
    shapes = [(0, 64, 1), (1, 0, 1), (1, 64, 0), (-1, 64, 1), (1, 64, 65536), (32768, 64, 1),
              (1, 1 << 20, 2048)]
    for B, T, H in shapes:
        assert L.fp8attn_prep(16, 16, 16, B, T, H, 128, None, 1, ctypes.byref(pp), 16, 1 << 30, None) == 1, (B, T, H)
        assert L.fp8attn_fwd(ctypes.byref(pp), B, T, H, 128, None, None, 0, 0, ctypes.c_float(256),
                             ctypes.c_float(-0.35), ctypes.c_float(0), 1, 16, 16, 1 << 30, None) == 1, (B, T, H)


def test_tail_plan(L):
    """Last-wave split plan (host only): split only a last wave of at most half
    the SMs; P = min(4, num_sms / n_tail) parts whose inner bounds are
    multiples of 4, strictly increasing, and balanced for max-only steps at
    half the cost of full ones."""
    import bit_attention_video_e4m3_gb300 as fa
    assert fa.tail_plan(1, 32760, 12, 152) == (4, 32, [0, 136, 204, 240, 256])     # Wan2.1 shape
    assert fa.tail_plan(1, 75600, 40, 152)[0] == 1        # last wave 80 of 152: kept whole
    assert fa.tail_plan(1, 1024, 8, 152)[0] == 1          # a single wave
    assert fa.tail_plan(1, 1024, 19, 152)[0] == 1         # whole waves only
    for B, T, H, sms in [(1, 1000, 3, 10), (1, 4000, 2, 20), (2, 5000, 7, 37), (1, 32760, 12, 148),
                         (3, 12345, 5, 100), (1, 300, 40, 7)]:
        parts, nt, lo = fa.tail_plan(B, T, H, sms)
        nv = -(-T // 128)
        total = B * H * nv
        ws = fa.fwd_tail_workspace_bytes(B, T, H, sms)
        if parts == 1:
            assert nt == 0 and lo == [] and ws == 256
            continue
        assert nt == total % sms and 0 < 2 * nt <= sms and total > sms
        assert 2 <= parts <= min(4, sms // nt)
        assert lo[0] == 0 and lo[-1] == nv and all(a < b for a, b in zip(lo, lo[1:]))
        assert all(x % 4 == 0 for x in lo[:-1])
        cost = [0.5 * lo[p] + (lo[p + 1] - lo[p]) for p in range(parts)]
        assert max(cost) - min(cost) <= 6, cost
        rows = parts * nt * 128
        assert ws == -(-(256 + rows * 8) // 16) * 16 + rows * 128 * 4
    assert fa.fwd_tail_workspace_bytes(1, 64, 1, 0) == 0
    from bit_attention_video_e4m3_gb300._lib import _Prepped
    pp = _Prepped(16, 16, 16, 16, 16, 16, 16)
    # num_sms < 1 and an empty shape are argument errors before any CUDA call
    assert L.fp8attn_fwd_tail_split(ctypes.byref(pp), 1, 64, 1, 128, 0, 0, ctypes.c_float(256),
                                    ctypes.c_float(-0.35), ctypes.c_float(0), 1, 0, 16, 16, 1 << 20, None) == 1
    assert L.fp8attn_fwd_tail_split(ctypes.byref(pp), 1, 0, 1, 128, 0, 0, ctypes.c_float(256),
                                    ctypes.c_float(-0.35), ctypes.c_float(0), 1, 152, 16, 16, 1 << 20, None) == 1


def test_cluster_bad_arguments_rejected(L):
    ws = L.fp8attn_cluster_workspace_bytes(1, 64, 1, 8)
    call = lambda v, D, K, r, it, perm, lab, wsb: L.fp8attn_v_cluster(v, 1, 64, 1, D, K, r, it, perm, lab,
                                                                     16, wsb, None)
    assert call(16, 64, 8, 8, 2, 16, None, ws) == 1          # D != 128
    assert call(None, 128, 8, 8, 2, 16, None, ws) == 1       # null V
    assert call(16, 128, 8, 8, 2, None, None, ws) == 1       # null perm
    assert call(16, 128, 0, 8, 2, 16, None, ws) == 1         # no clusters
    assert call(16, 128, 65, 8, 2, 16, None, ws) == 1        # too many clusters
    assert call(16, 128, 8, 17, 2, 16, None, ws) == 1        # too many dimensions
    assert call(16, 128, 8, 8, -1, 16, None, ws) == 1        # negative iterations
    assert call(24, 128, 8, 8, 2, 16, None, ws) == 1         # misaligned V
    assert call(16, 128, 8, 8, 2, 18, None, ws) == 1         # misaligned perm
    assert call(16, 128, 8, 8, 2, 16, 18, ws) == 1           # misaligned labels
    assert call(16, 128, 8, 8, 2, 16, None, ws - 16) == 5    # workspace too small


def test_split_helpers_and_bad_split_arguments(L):
    from bit_attention_video_e4m3_gb300._lib import _Prepped
    assert L.fp8attn_fwd_split_workspace_bytes(1, 1024, 2, 1) == L.fp8attn_fwd_workspace_bytes(1, 1024, 2)
    assert L.fp8attn_fwd_split_workspace_bytes(1, 1024, 2, 4) >= 4 * 2 * 1024 * (8 + 512)
    assert L.fp8attn_fwd_split_workspace_bytes(1, 1024, 2, 17) == 0
    # auto rule: all parts in one wave, at least 8 key tiles per part, at most 16 parts
    assert L.fp8attn_fwd_auto_splits(1, 32760, 12, 152) == 1
    assert L.fp8attn_fwd_auto_splits(1, 1024, 2, 152) == 1          # 8 key tiles: too short to split
    assert L.fp8attn_fwd_auto_splits(1, 4096, 1, 152) == 4          # 32 query tiles, 32 key tiles
    assert L.fp8attn_fwd_auto_splits(1, 4096, 2, 152) == 2          # 64 query tiles
    assert L.fp8attn_fwd_auto_splits(1, 8192, 1, 152) == 2
    assert L.fp8attn_fwd_auto_splits(1, 8192, 2, 152) == 1          # 128 query tiles: two would need 2 waves
    assert L.fp8attn_fwd_auto_splits(1, 2048, 1, 152) == 2          # 16 key tiles -> parts of 8
    assert L.fp8attn_fwd_auto_splits(1, 65536, 1, 152) == 1
    assert L.fp8attn_fwd_auto_splits(1, 128, 1, 152) == 1
    assert L.fp8attn_fwd_auto_splits(1, 131072, 1, 2000) == 1       # 1024 query tiles
    assert L.fp8attn_fwd_auto_splits(1, 16384, 1, 4096) == 16       # capped at 16
    pp = _Prepped(16, 16, 16, 16, 16, 16, 16)
    base = [ctypes.byref(pp), 1, 1024, 2, 128, None, None, 0, 0, ctypes.c_float(256), ctypes.c_float(-0.35),
            ctypes.c_float(0), 1]
    ws = L.fp8attn_fwd_split_workspace_bytes(1, 1024, 2, 4)
    assert L.fp8attn_fwd_split(*base, 0, 16, 16, ws, None) == 1         # n_splits < 1
    assert L.fp8attn_fwd_split(*base, 17, 16, 16, ws, None) == 1        # n_splits > 16
    assert L.fp8attn_fwd_split(*base, 4, 16, 16, ws - 16, None) == 5    # workspace too small


def test_prep_ex_argument_checks(L):
    from bit_attention_video_e4m3_gb300._lib import _Prepped
    ws = L.fp8attn_prep_workspace_bytes(1, 64, 1)
    full = _Prepped(16, 16, 16, 16, 16, 16, 16, None, 16, 16)
    no_v4 = _Prepped(16, 16, 16, 16, 16, 16, 16, None, None, None)
    args = lambda pp, vb, vf: (16, 16, 16, 1, 64, 1, 128, None, 1, 0, vb, vf, ctypes.byref(pp), 16, ws, None)
    assert L.fp8attn_prep_ex(*args(full, 0, 2)) == 1          # unknown V format
    assert L.fp8attn_prep_ex(*args(full, 1, 1)) == 1          # bias correction not offered with NVFP4
    assert L.fp8attn_prep_ex(*args(no_v4, 0, 1)) == 1         # NVFP4 without its outputs
    mis = _Prepped(16, 16, 16, 16, 16, 16, 16, None, 24, 16)
    assert L.fp8attn_prep_ex(*args(mis, 0, 1)) == 1           # misaligned v4


def test_selftest_argument_checks(L):
    assert L.fp8attn_selftest_wait_timeout(None, 1000000, None) == 5     # no workspace
    assert L.fp8attn_selftest_wait_timeout(24, 1000000, None) == 5       # misaligned workspace
    assert L.fp8attn_selftest_wait_timeout(16, 10, None) == 1            # limit below 100 us
    assert L.fp8attn_selftest_wait_timeout(16, 5 * 10**9, None) == 1     # limit above 1 s

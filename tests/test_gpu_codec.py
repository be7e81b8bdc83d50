"""The E4M3 conversion the kernels use (hardware cvt.rn.satfinite.e4m3x2.f32,
through fp8attn_e4m3_encode) against the oracle's encoder, value by value.

The rounding of an fp32 value to E4M3 depends on its sign, exponent, the
mantissa bits kept, the next bit and whether any lower bit is set.  The inputs
are every one of the 2^16 upper halves of an fp32 word (sign, exponent, top 7
mantissa bits: this is every bfloat16 value, so the prep's inputs scaled by a
power of two are covered exhaustively) combined with low halves that set none,
the lowest, a middle, the half-way and all of the remaining 16 mantissa bits,
plus random ones: every rounding case of every binade, ties included.
NaN inputs are left out (the encoder maps them to a NaN code, not a value).
The last test sweeps every one of the 2^32 fp32 bit patterns.
"""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from oracle import e4m3

pytestmark = pytest.mark.gpu


def _inputs():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    rng = np.random.default_rng(11)
    lows = [0x0000, 0x0001, 0x0100, 0x7FFF, 0x8000, 0x8001, 0xFFFF] + list(rng.integers(0, 1 << 16, 3))
    bits = (hi[:, None] | np.array(lows, dtype=np.uint32)[None, :]).ravel()
    x = bits.view(np.float32)
    return x[~np.isnan(x)]


def test_hardware_conversion_matches_the_oracle_encoder():
    x = _inputs()
    assert x.size > 600_000
    got = fa.e4m3_encode(torch.from_numpy(x).cuda()).cpu().numpy()
    want = e4m3.encode(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), hex(x[i:i + 1].view(np.uint32)[0]), got[i], want[i]) for i in bad[:8]]


def test_conversion_of_special_values():
    x = np.array([0.0, -0.0, 448.0, -448.0, 464.0, 480.0, 1e30, -np.inf, np.inf,
                  2.0 ** -9, 2.0 ** -10, -2.0 ** -10, 2.0 ** -10 * 1.0000001], dtype=np.float32)
    got = fa.e4m3_encode(torch.from_numpy(x).cuda()).cpu().numpy()
    assert list(got) == [0x00, 0x80, 0x7E, 0xFE, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0x01, 0x00, 0x80, 0x01]
    assert np.array_equal(got, e4m3.encode(x))


def test_odd_length_and_empty():
    x = torch.tensor([1.0, 2.0, 3.0], dtype=torch.float32, device="cuda")
    assert fa.e4m3_encode(x).cpu().tolist() == [0x38, 0x40, 0x44]
    assert fa.e4m3_encode(torch.empty(0, dtype=torch.float32, device="cuda")).numel() == 0


CHUNK = 1 << 24


@pytest.mark.slow
def test_every_fp32_pattern_matches_the_oracle_encoder():
    """All 2^32 fp32 bit patterns (NaN patterns excluded) through
    fp8attn_e4m3_encode, chunk by chunk, against the oracle's encoder computed
    by a spawn process pool on the host cores: zero mismatches."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os

    from tests import _codec_sweep

    n_chunks = (1 << 32) // CHUNK
    workers = max(1, min(16, len(os.sched_getaffinity(0))))
    mismatches, checked = 0, 0
    first_bad = []
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        futs = ex.map(_codec_sweep.oracle_chunk, [(c * CHUNK, (c + 1) * CHUNK) for c in range(n_chunks)])
        for c, want in enumerate(futs):
            lo = c * CHUNK
            start = lo if lo < (1 << 31) else lo - (1 << 32)        # the same 32 bits as int32
            bits = torch.arange(start, start + CHUNK, dtype=torch.int32, device="cuda")
            x = bits.view(torch.float32)
            got = fa.e4m3_encode(x).cpu().numpy()
            nan = torch.isnan(x).cpu().numpy()
            bad = np.nonzero((got != want) & ~nan)[0]
            mismatches += bad.size
            checked += int((~nan).sum())
            if bad.size and len(first_bad) < 8:
                first_bad += [(hex(lo + int(i)), int(got[i]), int(want[i])) for i in bad[:8]]
    assert checked == (1 << 32) - 2 * ((1 << 23) - 1)      # every non-NaN pattern
    assert mismatches == 0, first_bad

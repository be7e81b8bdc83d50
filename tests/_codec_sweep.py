"""Pool worker of the exhaustive E4M3 codec sweep (numpy and the oracle only,
so that spawned workers start quickly).  Test infrastructure."""
import numpy as np

from oracle import e4m3


def oracle_chunk(bounds):
    """Oracle E4M3 codes of the fp32 bit patterns [lo, hi) (uint8; NaN patterns
    give the NaN code and are masked out by the caller)."""
    lo, hi = bounds
    bits = np.arange(lo, hi, dtype=np.uint64).astype(np.uint32)
    with np.errstate(invalid="ignore"):
        return e4m3.encode(bits.view(np.float32))

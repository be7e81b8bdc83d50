"""The P-collapse effect on the GPU kernel (P-Cast Precision review, sections
3-5): with a few sink keys far above the rest, forward order at S = 1 casts
the non-sink probabilities against the sinks' maximum and most of them
underflow to code 0, so the output loses the non-sink mass; S = 256 lifts
them back into the E4M3 range, and reverse order casts them before the sinks
are seen.  Measured here as the relative error of the GPU output against
exact fp64 attention on sampled rows."""
import numpy as np
import pytest

from bit_attention_video_e4m3_gb300.workloads import make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu


def _err(delta, S, reverse, rows):
    w = make_workload("pcollapse", device="cuda", delta=delta, S=S, reverse=reverse)
    _, out, status = P.run_gpu(w)
    assert status == 0
    errs = []
    for h in (0, 5):
        ref = P.oracle_prep_head(w, 0, h)
        exact = P.exact_attention(w, ref, rows)
        errs.append(P.rel_l2(P.gpu_rows(out, 0, h, rows), exact))
    return float(np.mean(errs))


@pytest.mark.parametrize("delta", [6.0, 8.0])
def test_forward_s1_collapses_and_s256_or_reverse_recovers(delta):
    rows = P.sample_rows(16384, 96, seed=4)
    e = {(S, rev): _err(delta, S, rev, rows) for S in (1.0, 256.0, 448.0) for rev in (False, True)}
    print(f"delta={delta}: " + ", ".join(f"{'rev' if r else 'fwd'} S={int(S)}: {v:.4f}" for (S, r), v in e.items()))
    best = min(e.values())
    assert e[(1.0, False)] > 3 * e[(256.0, False)]           # the collapse, and its cure by S = 256
    assert e[(1.0, True)] < 1.5 * best                       # reverse order avoids it at any S
    assert e[(256.0, False)] < 1.5 * best and e[(256.0, True)] < 1.5 * best

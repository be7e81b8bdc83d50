"""Failure detection on the GPU without a fault: a bounded wait that nothing
ends must give up after its limit, report FP8ATTN_ERR_DEVICE_TIMEOUT through
the workspace status word, and leave the context usable (a normal prep and
attention afterwards still match the oracle)."""
import time

import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_a_timeout_and_the_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert fa.check_status(ws) == 0
    limit_ns = 20_000_000                                   # 20 ms
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fa.selftest_wait_timeout(ws, limit_ns)
    code = fa.check_status(ws)                              # synchronises
    dt = time.perf_counter() - t0
    assert code == 4                                        # FP8ATTN_ERR_DEVICE_TIMEOUT
    assert dt >= 0.02
    assert fa.check_status(ws) == 0                         # reading the status clears it
    # the context is still usable: a normal call matches the oracle
    w = make_workload("tiny", device="cuda", T=300, H=1, seed=71)
    pp, out, status = P.run_gpu(w)
    assert status == 0
    ref = P.oracle_prep_head(w, 0, 0)
    P.assert_prep_bitexact(pp, ref, 0, 0)
    rows = np.arange(w.T)
    assert P.rel_l2(P.gpu_rows(out, 0, 0, rows), P.oracle_attention(w, ref, rows)) <= P.REL_L2_TOL

"""Maximum-size case: a problem whose tensors hold more than 2^31 elements
(B=1, T=131072, H=136: 2.28 G elements per tensor, 13.7 GB of bf16 Q/K/V), so
every index and TMA stride beyond 32 bits is exercised.  Prep outputs are
checked bit for bit and attention rows within the tolerance on the first and
last head, in the first, a middle and the last query tile."""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import make_workload
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_more_than_2_31_elements():
    T, H = 131072, 136
    assert T * H * 128 > 2 ** 31
    w = make_workload("tiny", device="cuda", T=T, H=H, seed=70)
    pp, out, status = P.run_gpu(w)
    assert status == 0
    rows = np.concatenate([np.arange(0, 128, 5), np.arange(65536, 65536 + 128, 7), np.arange(T - 128, T, 3)])
    for h in (0, 135):
        ref = P.oracle_prep_head(w, 0, h)
        P.assert_prep_bitexact(pp, ref, 0, h)
        got = P.gpu_rows(out, 0, h, rows)
        o_ref = P.oracle_attention(w, ref, rows)
        assert P.rel_l2(got, o_ref) <= P.REL_L2_TOL
    del pp, out, w
    torch.cuda.empty_cache()

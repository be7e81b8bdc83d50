"""The error decomposition of the VC-Attention news article, section 1:
O - Oq = (P - Pq) V + Pq (V - Vq), the first term from quantising the
probabilities (and Q/K), the second from quantising V.  On the Wan2.2-shaped
recipe (clustered V with x20 outlier rows) V-Smooth (block means removed before
quantising, tokens in cluster order) shrinks the V term and the total error.
The article reports the V term at 82 % of the output error on real Wan2.2
activations; on these synthetic N(0,1) queries and keys the first term, which
also carries the E4M3 error of Q and K, is the larger one, so the share itself
is reported, not pinned."""
import math

import numpy as np

from bit_attention_video_e4m3_gb300.workloads import make_workload
from oracle import attention as A
from oracle import closed_forms as cf
from oracle import prep
from tests import parity as P


def _shares(vsmooth: bool):
    w = make_workload("wan22", device="cpu", T=4096, H=1)
    w.vsmooth = vsmooth
    ref = P.oracle_prep_head(w, 0, 0, vsmooth=vsmooth)
    rows = P.sample_rows(w.T, 160, seed=9)
    _, diag = A.emulated_attention_head(ref["qc"], ref["sq"], ref["kc"], ref["sk"], ref["vq"], ref["sv"],
                                        ref["mean"], w.T, rows, pcast=w.pcast, S=w.S, beta=w.beta,
                                        want_weights=True)
    Pq = np.stack([diag["weights"][int(r)] for r in rows])          # keys in permuted order
    perm = ref["perm"]
    k, v = ref["k"][perm], ref["v"][perm]
    X = (ref["q"][rows] @ k.T) / math.sqrt(128)
    Pe = np.exp(X - X.max(axis=1, keepdims=True))
    Pe /= Pe.sum(axis=1, keepdims=True)
    Vq = A.vtilde(ref["vq"], ref["sv"], ref["mean"], w.T)
    total, pterm, vterm = cf.decomposition(Pe, Pq, v, Vq)
    ep, ev = float(np.sum(pterm ** 2)), float(np.sum(vterm ** 2))
    return ep, ev, float(np.sum(total ** 2))


def test_v_smooth_shrinks_the_v_term():
    ep0, ev0, et0 = _shares(False)
    ep1, ev1, et1 = _shares(True)
    s0, s1 = ev0 / (ep0 + ev0), ev1 / (ep1 + ev1)
    print(f"V-term energy share: {s0:.3f} plain, {s1:.3f} with V-Smooth; "
          f"output error energy {et0:.4g} -> {et1:.4g}")
    assert ev1 < 0.75 * ev0              # V-Smooth removes a good part of the V term
    assert et1 < et0 and abs(ep1 - ep0) < 0.1 * ep0   # ... and leaves the P term alone

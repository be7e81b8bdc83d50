"""Closed forms of the P-cast study and the error decomposition (test infrastructure only).

P-Cast Precision review ("FP8 P-Cast Precision in Attention: Sink-Induced
Collapse and the Optimality of S=2^8"), section 3:
  * underflow: a probability p cast with static scale S becomes code 0 when
    p * S < 2^-10; with p = exp(s - m) that is s < m - 10 ln 2 - ln S
    (10 ln 2 = 6.93);
  * Proposition 1: with k sink keys of logit offset Delta, the running max is
    m = Delta + delta_k (delta_k = expected max of k standard normals,
    delta_4 ~= 1.03) and the non-sink underflow fraction is
    F(Delta, S) = Phi(Delta + delta_k - 6.93 - ln S);
  * Theorem 6: dp(S), the E4M3 quantisation step at the top of the scaled
    range relative to S, equals 2^-4 at every S = 2^k (k = 0..8) and exceeds
    it elsewhere; dp(S) = 2^(ceil(log2 S) - 4) / S;
  * Theorem 4: in reverse order with S = 256 the running max before the sink
    block is the max m of the non-sink logits and
    Pr[underflow] = Phi(m - 12.48) (12.48 = 18 ln 2).
VC-Attention news article, section 1: O - Oq = (P - Pq) V + Pq (V - Vq).
"""
from __future__ import annotations

import math

import numpy as np
from scipy import integrate

from .e4m3 import decode_table

LN2 = math.log(2.0)


def phi_cdf(x):
    """Standard normal CDF."""
    return 0.5 * math.erfc(-x / math.sqrt(2.0))


def _normal_pdf(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def max_of_k_pdf(x: float, k: int) -> float:
    """Density of the max of k iid standard normals: k phi(x) Phi(x)^(k-1)."""
    return k * _normal_pdf(x) * phi_cdf(x) ** (k - 1)


def delta_k(k: int) -> float:
    """Expected maximum of k iid standard normals (numerical quadrature)."""
    val, _ = integrate.quad(lambda x: x * max_of_k_pdf(x, k), -12, 12, limit=200)
    return val


def underflow_threshold(S: float) -> float:
    """s underflows when s < m - underflow_threshold(S); equals 10 ln 2 + ln S."""
    return 10.0 * LN2 + math.log(S)


def underflow_fraction_plugin(delta: float, S: float, k: int = 4) -> float:
    """Proposition 1 as printed: Phi(Delta + delta_k - 10 ln 2 - ln S)."""
    return phi_cdf(delta + delta_k(k) - underflow_threshold(S))


def underflow_fraction_averaged(delta: float, S: float, k: int = 4) -> float:
    """Proposition 1 with the running max averaged over its distribution.

    m = Delta + M, M the max of k standard normals; the fraction of non-sink
    logits s ~ N(0,1) below m - 10 ln 2 - ln S, averaged over M.
    """
    thr = underflow_threshold(S)
    val, _ = integrate.quad(lambda x: max_of_k_pdf(x, k) * phi_cdf(delta + x - thr),
                            -12, 12, limit=200)
    return val


def reverse_order_bound(m: float) -> float:
    """Theorem 4: Pr[underflow] = Phi(m - 18 ln 2) for reverse order with S = 256."""
    return phi_cdf(m - 18.0 * LN2)


def dp_closed_form(S: float) -> float:
    """Theorem 6 sawtooth: 2^(ceil(log2 S) - 4) / S."""
    return 2.0 ** (math.ceil(math.log2(S)) - 4) / S


def dp_brute_force(S: float) -> float:
    """E4M3 grid gap at the top of the scaled range [0, S], divided by S.

    The gap is between the largest code value strictly below S and the
    smallest code value at or above S, found by scanning the 256-entry table.
    """
    vals = decode_table()
    vals = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    below = vals[vals < S].max()
    above = vals[vals >= S]
    if above.size == 0:
        raise ValueError("S above the E4M3 range")
    return float(above.min() - below) / S


def decomposition(P: np.ndarray, Pq: np.ndarray, V: np.ndarray, Vq: np.ndarray):
    """Split the output error O - Oq into the P term and the V term.

    Returns (O - Oq, (P - Pq) V, Pq (V - Vq)), all fp64.
    """
    O = P @ V
    Oq = Pq @ Vq
    return O - Oq, (P - Pq) @ V, Pq @ (V - Vq)

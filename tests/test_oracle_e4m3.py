"""Pins of the oracle's E4M3 codec, ExpCast map and dp(S) sawtooth.

Each check compares the oracle with something other than itself: the format
facts the pages state, a brute-force nearest-value search over the code
table, torch's float8_e4m3fn conversion (a library routine), and closed forms.
"""
import math

import numpy as np
import pytest
import torch

from oracle import closed_forms as cf
from oracle import e4m3
from oracle.attention import PCAST_EXP2_CVT, PCAST_EXPCAST, pcast_codes


def _brute_force_encode(x):
    """Nearest finite E4M3 value by exhaustive search; ties to the even code; satfinite."""
    table = e4m3.decode_table()
    codes = np.arange(128)
    vals = table[:127]                      # 0x00..0x7E, the finite non-negative codes
    a = np.minimum(np.abs(x.astype(np.float64)), 448.0)
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among tied candidates prefer the even code (LSB of mantissa 0)
    even = cand & (codes[None, :127] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    out = codes[pick].astype(np.uint8)
    return np.where(np.signbit(x), out | 0x80, out).astype(np.uint8)


def test_table_format_facts():
    t = e4m3.decode_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.nanmax(t) == 448.0
    pos = t[:127]
    assert pos[1] == 2.0 ** -9                          # smallest subnormal
    assert np.all(np.diff(pos[:9]) == 2.0 ** -9)        # subnormal spacing
    for e in range(-6, 9):                              # 8 values per normal binade
        n = np.sum((pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1)))
        assert n == (7 if e == 8 else 8), e             # 480 is the NaN slot in E4M3FN
    # relative step inside a binade is 1/8 of its lower edge (12.5 %)
    for e in range(-6, 8):
        b = pos[(pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1))]
        assert np.allclose(np.diff(b) / 2.0 ** e, 0.125)


def _probe_values(rng):
    t = e4m3.decode_table()[:127]
    mids = 0.5 * (t[:-1] + t[1:])
    vals = [t, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
            np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
            2.0 ** rng.uniform(-14, 9.5, 200000),
            np.array([0.0, 2 ** -10, 2 ** -11, 464.0, 480.0, 1e6, 447.99])]
    x = np.concatenate(vals).astype(np.float32)
    sign = rng.random(x.size) < 0.5
    return np.where(sign, -x, x).astype(np.float32)


def test_encode_matches_brute_force():
    rng = np.random.default_rng(1)
    x = _probe_values(rng)
    got = e4m3.encode(x)
    want = _brute_force_encode(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_encode_matches_torch_float8_in_range():
    rng = np.random.default_rng(2)
    x = _probe_values(rng)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3.encode(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_decode_inverts_encode_on_every_code():
    t = e4m3.decode_table()
    finite = np.nonzero(np.isfinite(t))[0]
    assert np.array_equal(e4m3.encode(t[finite].astype(np.float32)), finite.astype(np.uint8))


def test_underflow_condition():
    # P-Cast review, section 3: p*S underflows to code 0 exactly when p*S < 2^-10
    for S in (1.0, 256.0, 448.0):
        p_under = np.float32(2.0 ** -10 / S * 0.999)
        assert e4m3.encode(np.float32(p_under * S)) == 0
    assert e4m3.encode(np.float32(2.0 ** -10)) == 0                       # tie -> even (0)
    assert e4m3.encode(np.float32(2.0 ** -10 * (1 + 2 ** -20))) == 1


def test_dp_sawtooth():
    # Theorem 6: dp(2^k) = 2^-4 for k = 0..8; larger for every other S
    for k in range(9):
        assert cf.dp_brute_force(2.0 ** k) == 2.0 ** -4
    for S in np.linspace(1.01, 447.9, 997):
        bf = cf.dp_brute_force(float(S))
        assert math.isclose(bf, cf.dp_closed_form(float(S)), rel_tol=1e-12), S
        if abs(math.log2(S) - round(math.log2(S))) > 1e-9:
            assert bf > 2.0 ** -4
    assert math.isclose(cf.dp_brute_force(448.0), 32.0 / 448.0)


def test_expcast_exact_at_powers_of_two():
    # c = round(8 z + 56 + beta): at integer z the code is 8z + 56, i.e. the
    # exact E4M3 code of 2^z (field layout: exponent z + 7, mantissa 0)
    for S in (1.0, 256.0):
        for z in range(-6, 9):
            p = 2.0 ** z / S
            if p > 1:
                continue
            c = pcast_codes(np.array([math.log(p)]), PCAST_EXPCAST, S, -0.35)[0]
            assert c == 8 * z + 56
            assert c == e4m3.encode(np.float32(2.0 ** z))
            assert e4m3.decode(c) == 2.0 ** z
    # S = 256, p = 2^-n -> code 120 - 8n
    for n in range(0, 15):
        c = pcast_codes(np.array([-n * math.log(2.0)]), PCAST_EXPCAST, 256.0, -0.35)[0]
        assert c == 120 - 8 * n


def test_expcast_within_one_code_of_rne():
    # over the normal range 8*log2(1+f) - 8f lies in [0, 0.69]; with beta=-0.35
    # the affine code differs from the round-to-nearest code by at most 1
    rng = np.random.default_rng(3)
    d = -rng.uniform(0, 14 * math.log(2.0), 200000)
    for S in (256.0, 448.0):
        ce = pcast_codes(d, PCAST_EXPCAST, S, -0.35).astype(int)
        cr = pcast_codes(d, PCAST_EXP2_CVT, S, -0.35).astype(int)
        normal = S * np.exp(d) >= 2.0 ** -6
        assert np.max(np.abs(ce - cr)[normal]) <= 1
        assert ce.max() <= 126

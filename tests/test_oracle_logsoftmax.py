"""Pins for the oracle's full-vocabulary log-softmax and float32 key rule.

The ranking comes from the output logits (zhiding.cn recsys-examples article,
section "语义ID：解决稀疏性与长尾问题"); the oracle turns a logit row into
log-probabilities with a full-vocabulary log-softmax.  Pinned here against
library routines (scipy, torch) and against the normalisation invariant.
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle.beam_search as obs
from oracle import log_softmax_row, ordered_f32


@pytest.mark.parametrize("seed,shift,std", [(0, 0.0, 2.0), (1, 900.0, 2.0), (2, -700.0, 30.0), (3, 0.0, 1e-3)])
def test_matches_scipy_and_torch(seed, shift, std):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(4096) * std + shift).astype(np.float32)
    lp, lse = log_softmax_row(x)
    ref = scipy.special.log_softmax(x.astype(np.float64))
    np.testing.assert_allclose(lp, ref, rtol=0, atol=1e-12 * max(1.0, abs(shift)))
    ref_t = torch.log_softmax(torch.from_numpy(x.astype(np.float64)), dim=0).numpy()
    np.testing.assert_allclose(lp, ref_t, rtol=0, atol=1e-12 * max(1.0, abs(shift)))
    assert abs(lse - scipy.special.logsumexp(x.astype(np.float64))) < 1e-12 * max(1.0, abs(shift))


def test_normalised_and_shift_invariant():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(151936) * 2.0
    lp, lse = log_softmax_row(x)
    assert abs(scipy.special.logsumexp(lp)) < 1e-12
    lp2, lse2 = log_softmax_row(x + 123.25)
    np.testing.assert_allclose(lp, lp2, atol=1e-9)
    assert abs(lse2 - lse - 123.25) < 1e-9


def test_uniform_row_closed_form():
    lp, lse = log_softmax_row(np.zeros(1024))
    np.testing.assert_allclose(lp, -np.log(1024.0), atol=1e-15)
    assert abs(lse - np.log(1024.0)) < 1e-15


def _round_f32(v: Fraction) -> np.float32:
    """Nearest IEEE-754 binary32 value of an exact rational, ties to even.

    Written from the format's definition (24-bit significand, normal
    exponents down to -126, subnormal quantum 2^-149), independently of numpy's
    own float32 conversion, so that the pin below does not restate the oracle.
    """
    if v == 0:
        return np.float32(0.0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()  # 2^e <= a < 2^(e+1) after the fix-up
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 23, -149)                 # value of the last significand bit
    m = a / Fraction(2) ** q
    n = m.numerator // m.denominator
    rest = m - n
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and n % 2 == 1):
        n += 1
    out = float(n * Fraction(2) ** q)     # n < 2^25: exact in float64 and in float32
    return np.float32(out if v > 0 else -out)


def _bits(v) -> int:
    return int(np.array([v], dtype=np.float32).view(np.uint32)[0])


def _key_triples(n, seed):
    """(S, x, LSE) at the workload's magnitudes: beam scores are sums of up to a few
    code log-probabilities, logits are 2*N(0,1), and the LSE of a 151936-entry row
    of such logits is about log(151936) + 2 = 13.9."""
    rng = np.random.default_rng(seed)
    S = (-rng.uniform(0.0, 40.0, n)).astype(np.float32)
    x = (rng.standard_normal(n) * 2.0).astype(np.float32)
    lse = (13.4 + rng.uniform(0.0, 1.0, n)).astype(np.float32)
    return S, x, lse


def test_key_f32_is_two_roundings_of_exact_values():
    # The key contract: key32 = fl32(S32 + fl32(x32 - LSE32)), each operation rounded
    # once.  Built here from exact rationals and the format's rounding rule; at least a
    # tenth of the triples must separate it from one rounding of the exact S + x - LSE
    # and from the other association fl32(fl32(S + x) - LSE), so that either mistake
    # in the oracle fails this test.
    S, x, lse = _key_triples(400, 11)
    n_one = n_assoc = 0
    for s, xi, li in zip(S, x, lse):
        fs, fx, fl = Fraction(float(s)), Fraction(float(xi)), Fraction(float(li))
        want = _round_f32(fs + Fraction(float(_round_f32(fx - fl))))
        k = obs.key_f32(s, xi, li)
        assert isinstance(k, np.float32)
        assert _bits(k) == _bits(want), (s, xi, li, k, want)
        n_one += _bits(_round_f32(fs + fx - fl)) != _bits(want)
        n_assoc += _bits(_round_f32(Fraction(float(_round_f32(fs + fx))) - fl)) != _bits(want)
    assert n_one >= 40 and n_assoc >= 40, (n_one, n_assoc)


def test_round_f32_matches_the_format_on_known_values():
    # the rounding helper itself: exact values, halfway cases (ties to even) and a
    # subnormal, each stated from the binary32 format
    assert _round_f32(Fraction(1)) == np.float32(1.0)
    ulp1 = Fraction(1, 2 ** 23)
    assert _bits(_round_f32(1 + ulp1 / 2)) == _bits(np.float32(1.0))              # tie -> even (1.0)
    assert _bits(_round_f32(1 + 3 * ulp1 / 2)) == _bits(np.float32(1.0)) + 2      # tie -> even (1 + 2 ulp)
    assert _bits(_round_f32(1 + ulp1 / 2 + Fraction(1, 2 ** 60))) == _bits(np.float32(1.0)) + 1
    assert _bits(_round_f32(Fraction(-3, 1))) == _bits(np.float32(-3.0))
    assert _bits(_round_f32(Fraction(1, 2 ** 149))) == 1                          # smallest subnormal
    assert _bits(_round_f32(Fraction(1, 2 ** 150))) == 0                          # tie below it -> 0 (even)
    assert _round_f32(Fraction(1, 10)) == np.float32(0.1)


def test_ordered_f32_is_monotone_and_merges_zeros():
    vals = np.array([-np.inf, -1e30, -2.5, -1e-40, -0.0, 0.0, 1e-40, 3.0, np.inf], dtype=np.float32)
    codes = [ordered_f32(v) for v in vals]
    assert codes[4] == codes[5]
    assert all(a < b for a, b in zip(codes[:4], codes[1:5]))
    assert all(a < b for a, b in zip(codes[5:], codes[6:]))

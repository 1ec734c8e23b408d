"""Pins for the oracle's full-vocabulary log-softmax and float32 key rule.

The ranking comes from the output logits (zhiding.cn recsys-examples article,
section "语义ID：解决稀疏性与长尾问题"); the oracle turns a logit row into
log-probabilities with a full-vocabulary log-softmax.  Pinned here against
library routines (scipy, torch) and against the normalisation invariant.
"""
import numpy as np
import pytest
import scipy.special
import torch

from oracle import key_f32, log_softmax_row, ordered_f32


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


def test_key_f32_rounds_each_operation():
    # S + (x - L) in float32, one rounding per operation; the fused or float64
    # evaluation differs for these values.
    s, x, l = np.float32(-3.1415927), np.float32(1.0000001), np.float32(13.987654)
    k = key_f32(s, x, l)
    assert k.dtype == np.float32
    d = np.float32(x - l)
    assert k == np.float32(s + d)
    exact = float(s) + (float(x) - float(l))
    assert abs(float(k) - exact) <= 2 * np.spacing(np.float32(abs(exact)))


def test_ordered_f32_is_monotone_and_merges_zeros():
    vals = np.array([-np.inf, -1e30, -2.5, -1e-40, -0.0, 0.0, 1e-40, 3.0, np.inf], dtype=np.float32)
    codes = [ordered_f32(v) for v in vals]
    assert codes[4] == codes[5]
    assert all(a < b for a, b in zip(codes[:4], codes[1:5]))
    assert all(a < b for a, b in zip(codes[5:], codes[6:]))

"""The inputs of the merge's multi-level parity cases (tests/test_zz_no_alloc.py) reach the
levels they are meant to reach.  The threshold search is restated here on the host: buckets of
2^sh values over [a0, largest key] (sh the smallest with (b - a) >> sh < 256), the bucket holding
the k-th largest key, bucketed again while it holds more than 1024 keys of more than one value;
a0 is the smallest row maximum when there are at least k rows.  Keys are the code logits (the
cases make every row's log-sum-exp 0 and the beam scores 0), as order-preserving uint32."""
import numpy as np
import pytest

from tests.test_zz_no_alloc import _level_rows


def _ordered(f):
    u = np.asarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)


def _levels(x, code_lo, n_codes, k, cap=1024):
    keys = _ordered(x[:, code_lo:code_lo + n_codes])
    flat = keys.reshape(-1)
    a = int(flat.min())
    if keys.shape[0] >= k:
        a = max(a, int(keys.max(axis=1).min()))
    b, kk, out = int(flat.max()), k, []
    for _ in range(4):
        span = (b - a) >> 8
        sh = int(span).bit_length()
        inr = flat[(flat >= a) & (flat <= b)]
        h = np.bincount(((inr - a) >> sh).astype(np.int64), minlength=256)
        above = 0
        for d in range(255, -1, -1):
            if above + h[d] >= kk:
                break
            above += int(h[d])
        kk -= above
        a = a + d * (1 << sh)
        b = min(b, a + (1 << sh) - 1)
        out.append((above, int(h[d])))
        if h[d] <= cap or a == b:
            break
    return out


@pytest.mark.parametrize("levels,n_rows,n_codes", [(2, 64, 128), (3, 64, 128), (3, 256, 1024)])
def test_level_cases_reach_their_levels(levels, n_rows, n_codes):
    x, code_lo, C = _level_rows(levels, n_rows=n_rows, n_codes=n_codes)
    steps = _levels(x, code_lo, C, 100)
    assert len(steps) == levels, steps
    # keys above the chosen bucket at every level (the per-warp counts add up across levels)
    assert all(above > 0 for above, _ in steps), steps
    # every level but the last holds more than 1024 keys; the last is ranked directly
    assert all(c > 1024 for _, c in steps[:-1]) and steps[-1][1] <= 1024, steps

"""Host-side invariants of the attention schedule (gr_attn_schedule): no GPU needed.

The decode attention kernel works through this table: every CTA runs its jobs in order, a
unit cut over several CTAs is finished by its first key range (the merger), and the later
ranges publish their partial results for it.  The kernel is correct only if
  - every key tile of every unit is covered exactly once, in order, by the unit's jobs;
  - a unit's jobs own consecutive piece slots, the first of which is the merger;
  - a later range of a cut unit is the FIRST job of its CTA (it publishes before it waits
    for anything) and the merger is the LAST job of its CTA;
  - the CTA ranges partition the job list in order.
These are checked over many random batch shapes, including degenerate ones.
"""
import math

import numpy as np
import pytest

from beam_decode_gb300 import binding as B

pytestmark = pytest.mark.skipif(
    not __import__("os").path.exists(B.LIB_PATH), reason="libgrbeam not built")

TILE_KEYS = 128
TILE_ROWS = 128
UNIT_ROWS = 256


def expected_units(G, n_kv, ctx_lens, widths):
    """Units in order: requests, KV heads, beam blocks of UNIT_ROWS / G beams."""
    bpu = UNIT_ROWS // G
    out = []
    for r, (T, W) in enumerate(zip(ctx_lens, widths)):
        tiles = math.ceil(T / TILE_KEYS)
        for h in range(n_kv):
            for b0 in range(0, W, bpu):
                rows = min(bpu, W - b0) * G
                out.append((r, h, b0, math.ceil(rows / TILE_ROWS), tiles))
    return out


def check_schedule(G, n_kv, ctx_lens, widths, n_sm, attn_kernel=0):
    """attn_kernel 0 (automatic) and 1: the single-CTA kernel's schedule (one entry per CTA);
    2: the CTA-pair kernel's, over n_sm / 2 pairs."""
    units, jobs, ctas = B.attn_schedule(G * n_kv, n_kv, ctx_lens, widths, n_sm, head_dim=128,
                                        attn_kernel=attn_kernel)
    exp = expected_units(G, n_kv, ctx_lens, widths)
    assert len(units) == len(exp)
    for u, e in zip(units, exp):
        assert (u[0], u[1], u[2], u[3], u[6]) == e
    tiles_all = sum(e[4] for e in exp)
    if attn_kernel == 2:
        assert len(ctas) == min(max(n_sm // 2, 1), tiles_all)
    else:
        assert len(ctas) == min(n_sm, tiles_all)
    # CTA ranges partition the job list in order
    assert ctas[0, 0] == 0 and ctas[-1, 1] == len(jobs)
    assert np.all(ctas[1:, 0] == ctas[:-1, 1]) and np.all(ctas[:, 1] >= ctas[:, 0])
    cta_of = np.empty(len(jobs), np.int64)
    for k, (a, b) in enumerate(ctas):
        cta_of[a:b] = k
    # a job's slot is its index; a unit's jobs are its slots, in key order, covering every tile once
    assert np.all(jobs[:, 3] == np.arange(len(jobs)))
    for ui, u in enumerate(units):
        first, n_slots, n_tiles = u[4], u[5], u[6]
        assert n_slots >= 1
        js = jobs[first:first + n_slots]
        assert np.all(js[:, 0] == ui)
        assert js[0, 1] == 0 and js[-1, 2] == n_tiles
        assert np.all(js[:, 2] > js[:, 1])
        assert np.all(js[1:, 1] == js[:-1, 2])
        if n_slots > 1:
            merger = first
            assert merger == ctas[cta_of[merger], 1] - 1, "the merger of a cut unit is its CTA's last job"
            for s in range(first + 1, first + n_slots):
                assert s == ctas[cta_of[s], 0], "a later range of a cut unit is its CTA's first job"
    # every job belongs to exactly one unit's slot range
    owner = np.full(len(jobs), -1)
    for ui, u in enumerate(units):
        assert np.all(owner[u[4]:u[4] + u[5]] == -1)
        owner[u[4]:u[4] + u[5]] = ui
    assert np.all(owner >= 0)
    return units, jobs, ctas


@pytest.mark.parametrize("G,n_kv", [(1, 8), (2, 8), (4, 2), (8, 1), (16, 1)])
def test_schedule_invariants_random_batches(G, n_kv):
    rng = np.random.default_rng([7, G, n_kv])
    width_choices = [1, 3, 16, 30, 32, 64, 100, 128, 200, 256, 300, 513, 1024]
    for trial in range(40):
        n_req = int(rng.integers(1, 33))
        ctx = rng.choice([1, 7, 128, 129, 500, 1000, 2000, 5000, 8191], size=n_req).astype(int)
        ctx = np.where(rng.random(n_req) < 0.3, rng.integers(1, 9000, size=n_req), ctx)
        widths = rng.choice(width_choices, size=n_req).astype(int)
        n_sm = int(rng.choice([1, 2, 7, 76, 148, 152]))
        check_schedule(G, n_kv, list(ctx), list(widths), n_sm)
        check_schedule(G, n_kv, list(ctx), list(widths), n_sm, attn_kernel=2)


def test_schedule_of_the_long_workload():
    """8 requests x ctx 5000 x beam 256, 16/8 heads on 152 SMs: 128 units of two tiles over
    40 key tiles; units are cut, and their pieces are first jobs."""
    units, jobs, ctas = check_schedule(2, 8, [5000] * 8, [256] * 8, 152)
    assert len(units) == 128 and np.all(units[:, 3] == 2) and np.all(units[:, 6] == 40)
    assert np.sum(units[:, 5] > 1) > 0
    assert len(ctas) == 152
    # a CTA runs at most two jobs here: a piece of one unit, then the merger of the next
    assert np.max(ctas[:, 1] - ctas[:, 0]) <= 2
    # the CTA-pair kernel: the same units over 76 CTA pairs
    units, jobs, ctas = check_schedule(2, 8, [5000] * 8, [256] * 8, 152, attn_kernel=2)
    assert len(ctas) == 76


def test_short_units_are_kept_whole_when_cuts_gain_little():
    """16 requests x ctx 1000 x beam 256: 256 units of 8 key tiles.  Whole units (two per CTA)
    give a bound within the cut penalty of the cut schedule, so no unit is cut and every unit
    is one job; the long workload (previous test) keeps its cuts."""
    units, jobs, ctas = check_schedule(2, 8, [1000] * 16, [256] * 16, 152)
    assert len(units) == 256 and np.all(units[:, 6] == 8)
    assert np.all(units[:, 5] == 1) and len(jobs) == 256
    assert np.max(ctas[:, 1] - ctas[:, 0]) == 2
    # the pair kernel's schedule still cuts where that balances its pairs
    check_schedule(2, 8, [1000] * 16, [256] * 16, 152, attn_kernel=2)


def test_kernel_choice_and_pair_kernel_limits():
    """The automatic choice is the single-CTA kernel; the pair kernel needs head_dim 128."""
    _, _, c0 = B.attn_schedule(16, 8, [5000] * 8, [256] * 8, 152, head_dim=128, attn_kernel=0)
    _, _, c1 = B.attn_schedule(16, 8, [5000] * 8, [256] * 8, 152, head_dim=128, attn_kernel=1)
    assert len(c0) == len(c1) == 152
    with pytest.raises(B.GrError) as e:
        B.attn_schedule(16, 8, [5000] * 8, [256] * 8, 152, head_dim=64, attn_kernel=2)
    assert e.value.status == B.GR_ERR_UNSUPPORTED
    with pytest.raises(B.GrError) as e:
        B.attn_schedule(16, 8, [5000] * 8, [256] * 8, 152, attn_kernel=3)
    assert e.value.status == B.GR_ERR_INVALID_ARG


def test_schedule_degenerate_batches():
    check_schedule(2, 8, [1], [1], 152)            # one key, one beam
    check_schedule(2, 8, [1], [1], 1)              # everything on one CTA
    check_schedule(16, 1, [8191], [1024], 3)       # widest beam, many units, few CTAs
    units, jobs, ctas = check_schedule(1, 1, [128 * 300], [1], 152)  # one unit cut over many CTAs
    assert len(units) == 1 and units[0, 5] > 1


def test_schedule_rejects_bad_arguments():
    with pytest.raises(B.GrError):
        B.attn_schedule(16, 8, [0], [256], 152)
    with pytest.raises(B.GrError):
        B.attn_schedule(16, 8, [100], [2000], 152)
    with pytest.raises(B.GrError):
        B.attn_schedule(24, 8, [100], [16], 152)   # 3 query heads per KV head
    with pytest.raises(B.GrError):
        B.attn_schedule(16, 8, [100], [16], 0)

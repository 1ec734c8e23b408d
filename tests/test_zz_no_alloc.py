"""gr_constrained_topk_noalloc: the constrained top-K for callers that cannot
allocate device memory (a plugin handed only its input and output tensors, a
service whose device memory is fixed at start-up).  Its scratch is a fixed
array inside the library.  Through the C ABI, these tests check:
  * two calls in a row give the selection of gr_constrained_topk on the same
    inputs, keys bit for bit;
  * against the CPU oracle's sort-based selection (float64 log-sum-exp, the
    float32 key contract, key descending then flat index ascending): ties
    that straddle the k-th key, fewer candidates than k, rows with a NaN
    logit, and the largest size the fixed scratch holds with k = 1024;
  * sizes beyond the fixed scratch are refused.

The oracle cases use logits on a grid of 1/8 and beam scores on a grid of
2^-12, every row holding the same values in another order: each row's
log-sum-exp is then the same number, so a last-bit difference between the
GPU's float32 log-sum-exp and the oracle's rounded float64 one moves no key
past another, and the selections must agree exactly.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

from beam_decode_gb300 import binding as B
from tests.harness import LP_TOL, LockStep, Spec

pytestmark = pytest.mark.gpu


def _call(x, ld, n_rows, vocab, code_lo, n_codes, scores, mask, k, outs):
    import torch
    p, c, key, n = outs
    return B.lib().gr_constrained_topk_noalloc(
        x.data_ptr(), ld, n_rows, vocab, code_lo, n_codes, None if scores is None else scores.data_ptr(),
        mask.data_ptr(), k, p.data_ptr(), c.data_ptr(), key.data_ptr(), n.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _outs(k):
    import torch
    return (torch.full((k,), -1, dtype=torch.int32, device="cuda"),
            torch.full((k,), -1, dtype=torch.int32, device="cuda"),
            torch.full((k,), float("nan"), device="cuda"),
            torch.full((1,), -1, dtype=torch.int32, device="cuda"))


def _run(x, scores, mask, code_lo, n_codes, k):
    """One call on host arrays; returns (parents, codes, keys) of the survivors."""
    import torch
    n_rows, vocab = x.shape
    dx = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    ds = None if scores is None else torch.from_numpy(scores.astype(np.float32)).cuda()
    dm = torch.from_numpy(np.ascontiguousarray(mask).view(np.int32)).cuda()
    outs = _outs(k)
    st = _call(dx, vocab, n_rows, vocab, code_lo, n_codes, ds, dm, k, outs)
    assert st == 0, B.lib().gr_last_error().decode()
    torch.cuda.synchronize()
    m = int(outs[3].item())
    assert 0 <= m <= k
    return outs[0].cpu().numpy()[:m], outs[1].cpu().numpy()[:m], outs[2].cpu().numpy()[:m]


def _oracle(x, scores, mask, code_lo, n_codes, k):
    """The oracle's selection: float64 LSE of each row rounded to float32, key32 = S + (x - LSE)
    rounded once per operation, candidates ordered by key descending then flat index ascending,
    the first min(k, #candidates).  Rows whose log-sum-exp is not finite (a NaN logit) give no
    candidates."""
    from oracle import key_f32, log_softmax_row
    from oracle.beam_search import rank_candidates
    n_rows = x.shape[0]
    cands = []
    for b in range(n_rows):
        lse = log_softmax_row(x[b].astype(np.float64))[1]
        if not np.isfinite(lse):
            continue
        codes = [c for c in range(n_codes) if (int(mask[b, c >> 5]) >> (c & 31)) & 1]
        if not codes:
            continue
        s = np.float32(0.0) if scores is None else np.float32(scores[b])
        keys = key_f32(np.full(len(codes), s, dtype=np.float32), x[b, code_lo + np.array(codes)],
                       np.full(len(codes), np.float32(lse), dtype=np.float32))
        for c, key in zip(codes, keys):
            cands.append((np.float32(0.0) if key == 0 else key, b * n_codes + c, b, c))
    sel = rank_candidates(cands)[:k]
    return (np.array([e[2] for e in sel], dtype=np.int32), np.array([e[3] for e in sel], dtype=np.int32),
            np.array([e[0] for e in sel], dtype=np.float32))


def _grid_rows(n_rows, vocab, code_lo, n_codes, seed, same_order=False):
    """Logit rows on a grid of 1/8: the non-code part is shared, the code part is a row-wise
    permutation of n_codes distinct grid values (so every row's log-sum-exp is the same)."""
    rng = np.random.default_rng(seed)
    base = (rng.integers(-40, 40, vocab) / 8.0).astype(np.float32)
    vals = (np.arange(n_codes) - n_codes // 2).astype(np.float32) / 8.0
    x = np.tile(base, (n_rows, 1))
    perm = rng.permutation(n_codes)
    for b in range(n_rows):
        x[b, code_lo:code_lo + n_codes] = vals[perm if same_order else rng.permutation(n_codes)]
    return x


def _full_mask(n_rows, n_codes):
    m = np.zeros((n_rows, (n_codes + 31) // 32), dtype=np.uint32)
    for c in range(n_codes):
        m[:, c >> 5] |= np.uint32(1) << np.uint32(c & 31)
    return m


def _assert_same(got, exp):
    gp, gc, gk = got
    ep, ec, ek = exp
    assert len(gp) == len(ep), (len(gp), len(ep))
    assert np.array_equal(gp, ep)
    assert np.array_equal(gc, ec)
    assert np.max(np.abs(gk - ek), initial=0.0) <= LP_TOL


def _level_rows(levels, seed=5, n_rows=64, n_codes=128):
    """Keys that make the merge bucket its threshold bucket again (the first level's bucket
    holds more than the 1024 keys it ranks directly, all distinct).  Every row's dominant
    logit sits outside the codes and the code logits are at most -100, so each row's
    log-sum-exp is 0 on the GPU and ~1e-43 in the oracle, and with zero beam scores every key
    is its code logit on both sides.  64 rows x 128 codes by default, k = 100: 40 keys far above, for three
    levels 30 more just above the band, 3000 consecutive float32 values (the band), the rest
    below (-199..-198.5 for two levels, -1e30 for three: a wider first level), and two rows
    of low keys only, so that the smallest row maximum leaves the band in range."""
    vocab, code_lo = 2 * max(512, n_codes), max(512, n_codes)
    rng = np.random.default_rng(seed)
    x = np.full((n_rows, vocab), -1000.0, dtype=np.float32)
    x[:, 0] = 0.0
    high = (-100.0 - 0.25 * np.arange(40)).astype(np.float32)
    mid = (-140.0 - 0.0625 * np.arange(30)).astype(np.float32) if levels == 3 else np.zeros(0, np.float32)
    band = np.empty(3000, dtype=np.float32)
    band[0] = -150.0
    for i in range(1, len(band)):
        band[i] = np.nextafter(band[i - 1], np.float32(0.0))
    special = np.concatenate([high, mid, band])
    n_main = (n_rows - 2) * n_codes
    low = np.float32(-199.0 if levels == 2 else -1e30)
    vals = np.full(n_main, low, dtype=np.float32)
    if levels == 2:
        vals = (low + 0.5 * rng.random(n_main)).astype(np.float32)
    vals[:len(special)] = special
    x[:n_rows - 2, code_lo:code_lo + n_codes] = vals[rng.permutation(n_main)].reshape(n_rows - 2, n_codes)
    x[n_rows - 2:, code_lo:code_lo + n_codes] = low
    return x, code_lo, n_codes


@pytest.mark.parametrize("levels,n_rows,n_codes", [(2, 64, 128), (3, 64, 128), (3, 256, 1024)])
def test_noalloc_threshold_bucketed_again(levels, n_rows, n_codes):
    # 256 x 1024 candidates: 32768 per CTA, more than its shared-memory stage, so every pass
    # re-reads the keys from global memory
    x, code_lo, C = _level_rows(levels, n_rows=n_rows, n_codes=n_codes)
    mask = _full_mask(x.shape[0], C)
    exp = _oracle(x, None, mask, code_lo, C, 100)
    assert len(exp[0]) == 100
    got = _run(x, None, mask, code_lo, C, 100)
    _assert_same(got, exp)
    assert np.array_equal(got[2].view(np.uint32), exp[2].view(np.uint32))  # keys bit for bit


def test_noalloc_all_keys_equal_in_shared_memory():
    """8192 candidates with one key value (constant logits): the first level's bucket is a
    single value holding more keys than are ranked directly, so the first k in flat order are
    taken, from the keys staged in shared memory."""
    n_rows, C, vocab, code_lo = 64, 128, 1024, 512
    x = np.zeros((n_rows, vocab), dtype=np.float32)
    mask = _full_mask(n_rows, C)
    exp = _oracle(x, None, mask, code_lo, C, 100)
    got = _run(x, None, mask, code_lo, C, 100)
    _assert_same(got, exp)
    assert np.array_equal(got[0], np.zeros(100, np.int32)) and np.array_equal(got[1], np.arange(100))


def test_noalloc_matches_constrained_topk_twice():
    import torch
    C = 256
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=64, vocab=4096, n_levels=2, codes_per_level=C,
                code_base=4096 - 2 * C, ctx_lens=[8], widths=[64], n_items=[20000], seed=41)
    ls = LockStep(spec)
    ls.topk_step()                                   # level 0 through the existing path
    beam = ls.beam
    _, tok0, _, sc0 = beam.path(0, 0)
    n = len(tok0)
    code0 = tok0 - spec.code_base
    items = ls.items[0]
    mask = np.zeros((n, C // 32), dtype=np.uint32)
    for b in range(n):
        for c in np.unique(items[items[:, 0] == code0[b], 1]):
            mask[b, c >> 5] |= np.uint32(1) << np.uint32(c & 31)
    x = torch.from_numpy(ls.logits(1)).cuda()
    ld = x.shape[1]
    # existing entry point at step 1 (its own log-sum-exp, as the no-alloc entry point)
    beam.constrained_topk(x)
    beam.advance()
    par1, tok1, _, sc1 = beam.path(0, 1)
    # the no-alloc entry point, twice, on the first n rows: the same selection, keys bit for bit
    dmask = torch.from_numpy(mask.view(np.int32)).cuda()
    dscore = torch.from_numpy(sc0.astype(np.float32)).cuda()
    k = spec.widths[0]
    for _ in range(2):
        outs = _outs(k)
        st = _call(x, ld, n, spec.vocab, spec.code_base + C, C, dscore, dmask, k, outs)
        assert st == 0, B.lib().gr_last_error().decode()
        torch.cuda.synchronize()
        m = int(outs[3].item())
        assert m == len(par1)
        assert np.array_equal(outs[0].cpu().numpy()[:m], par1)
        assert np.array_equal(outs[1].cpu().numpy()[:m], tok1 - spec.code_base - C)
        assert np.array_equal(outs[2].cpu().numpy()[:m].view(np.uint32), sc1.view(np.uint32))


@pytest.mark.parametrize("k", [100, 40])
def test_noalloc_ties_straddle_the_kth_key(k):
    # identical rows and scores: every code's key is tied across all 12 rows, and k = 100
    # (8 * 12 + 4) or 40 (3 * 12 + 4) cuts a tie group, so the last four survivors come from the
    # flat order; with k = 40 < 64 codes each row keeps only its own top 40 first (stage 1)
    n_rows, vocab, C, code_lo = 12, 1024, 64, 512
    x = _grid_rows(n_rows, vocab, code_lo, C, seed=3, same_order=True)
    scores = np.zeros(n_rows, dtype=np.float32)
    mask = _full_mask(n_rows, C)
    exp = _oracle(x, scores, mask, code_lo, C, k)
    assert len(set(exp[1][-4:].tolist())) == 1 and exp[0][-4:].tolist() == [0, 1, 2, 3]  # the cut tie group
    for _ in range(2):
        _assert_same(_run(x, scores, mask, code_lo, C, k), exp)


def test_noalloc_fewer_candidates_than_k():
    n_rows, vocab, C, code_lo = 8, 1024, 256, 640
    x = _grid_rows(n_rows, vocab, code_lo, C, seed=4)
    scores = (-np.arange(n_rows) / 4096.0).astype(np.float32)
    mask = np.zeros((n_rows, C // 32), dtype=np.uint32)
    rng = np.random.default_rng(5)
    for b in range(n_rows):
        for c in rng.choice(C, 3, replace=False):
            mask[b, c >> 5] |= np.uint32(1) << np.uint32(c & 31)
    exp = _oracle(x, scores, mask, code_lo, C, 64)
    assert len(exp[0]) == 3 * n_rows
    _assert_same(_run(x, scores, mask, code_lo, C, 64), exp)


def test_noalloc_rows_with_a_nan_logit_give_no_candidates():
    n_rows, vocab, C, code_lo = 10, 1024, 128, 768
    x = _grid_rows(n_rows, vocab, code_lo, C, seed=6)
    x[2, 17] = np.nan               # outside the code range
    x[7, code_lo + 5] = np.nan      # inside it
    scores = (-np.arange(n_rows) / 4096.0).astype(np.float32)
    mask = _full_mask(n_rows, C)
    exp = _oracle(x, scores, mask, code_lo, C, 300)
    assert not ({2, 7} & set(exp[0].tolist()))
    _assert_same(_run(x, scores, mask, code_lo, C, 300), exp)


def test_noalloc_largest_scratch_and_k_1024_twice():
    # exactly GR_NOALLOC_MAX_CANDIDATES candidates (256 rows x 1024 codes), k = 1024
    n_rows, C = 256, 1024
    vocab, code_lo = 2048, 1024
    assert n_rows * C == B.GR_NOALLOC_MAX_CANDIDATES
    x = _grid_rows(n_rows, vocab, code_lo, C, seed=7)
    scores = (-np.arange(n_rows) / 4096.0).astype(np.float32)
    mask = _full_mask(n_rows, C)
    rng = np.random.default_rng(8)
    drop = rng.random((n_rows, C)) < 0.25       # a quarter of the codes are not valid
    for b, c in zip(*np.nonzero(drop)):
        mask[b, c >> 5] &= ~(np.uint32(1) << np.uint32(c & 31))
    exp = _oracle(x, scores, mask, code_lo, C, 1024)
    assert len(exp[0]) == 1024
    for _ in range(2):
        _assert_same(_run(x, scores, mask, code_lo, C, 1024), exp)


def test_noalloc_refuses_sizes_beyond_scratch():
    import torch
    x = torch.zeros((8, 1024), device="cuda")
    mask = torch.zeros((8, 32), dtype=torch.int32, device="cuda")
    outs = (torch.zeros(8, dtype=torch.int32, device="cuda"), torch.zeros(8, dtype=torch.int32, device="cuda"),
            torch.zeros(8, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"))
    too_many_rows = B.GR_NOALLOC_MAX_CANDIDATES // 1024 + 1
    assert _call(x, 1024, too_many_rows, 1024, 0, 1024, None, mask, 8, outs) == B.GR_ERR_CAPACITY
    assert _call(x, 1024, 8, 1024, 0, 1024, None, mask, 2048, outs) == B.GR_ERR_CAPACITY
    assert _call(x, 1024, 8, 1024, 0, 2048, None, mask, 8, outs) == B.GR_ERR_CAPACITY

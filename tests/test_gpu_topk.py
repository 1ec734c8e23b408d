"""gr_constrained_topk + gr_beam_advance against the oracle step.

Bit-exact selections / BeamPath under the float32 key contract (the oracle's
LSE passed as lse_in); with the GPU's own LSE: LSE and log-probabilities within
1e-4 and identical selections (no near-ties on these seeds).  Edge cases: exact
ties within and across beams, one valid code per prefix, width above the number
of candidates, width 1, 1024-wide beams, vocab rows with padding.
"""
import numpy as np
import pytest

from tests.harness import LP_TOL, LockStep, Spec

pytestmark = pytest.mark.gpu


def test_default_lse_mode_tolerances():
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=64, vocab=151936, n_levels=3, codes_per_level=256,
                code_base=151936 - 768, ctx_lens=[8, 8, 8], widths=[256, 100, 33], n_items=[50000] * 3, seed=21)
    ls = LockStep(spec)
    r = ls.topk_step(lse_mode=False)
    assert r["lse_err"] <= LP_TOL and r["lp_err"] <= LP_TOL, r
    assert not r["mismatch"], r
    ls2 = LockStep(spec)
    ls2.topk_step(lse_mode=True)
    r = ls2.topk_step(lse_mode=False)
    assert r["lse_err"] <= LP_TOL and r["lp_err"] <= LP_TOL, r
    assert not r["mismatch"], r


def _ties(ls, t, x):
    # exact ties: quantised logits, and duplicate rows for pairs of beams
    x = np.round(x * 2.0) / 2.0
    rows = ls.beam.rows
    for b in range(0, rows - 1, 2):
        x[b + 1] = x[b]
    return x


@pytest.mark.parametrize("W", [1, 5, 64, 256])
def test_exact_ties(W):
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=64, vocab=4096, n_levels=3, codes_per_level=64,
                code_base=4096 - 192, ctx_lens=[8, 8], widths=[W, W], n_items=[5000, 5000], seed=22 + W)
    ls = LockStep(spec, logits_fn=_ties)
    for t in range(3):
        r = ls.topk_step(lse_mode=True)
        assert not r["mismatch"], (t, r)


def test_one_child_per_prefix():
    # every item has a unique first code: after level 0 each beam has one valid code
    C = 64
    items = np.stack([np.arange(C), np.random.default_rng(0).integers(0, C, C)], axis=1).astype(np.int32)
    spec = Spec(vocab=1024, n_levels=2, codes_per_level=C, code_base=512, widths=[16], n_items=[C], seed=23)
    ls = LockStep.__new__(LockStep)
    import tests.harness as H
    orig = H.make_items
    H.make_items = lambda s: [items]
    try:
        ls.__init__(spec)
    finally:
        H.make_items = orig
    for t in range(2):
        r = ls.topk_step(lse_mode=True)
        assert not r["mismatch"], (t, r)
        assert r["n_sel"] == [16]


def test_wide_beam_1024():
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=64, vocab=8192, n_levels=2, codes_per_level=512,
                code_base=8192 - 1024, ctx_lens=[4], widths=[1024], n_items=[200000], seed=24)
    ls = LockStep(spec)
    for t in range(2):
        r = ls.topk_step(lse_mode=True)
        assert not r["mismatch"], (t, r)
        assert r["n_sel"][0] == min(1024, r["n_sel"][0])


def test_single_level_catalogue():
    spec = Spec(vocab=1024, n_levels=1, codes_per_level=100, code_base=0, widths=[10, 200],
                ctx_lens=[4, 4], n_items=[60, 60], seed=25)
    ls = LockStep(spec)
    r = ls.topk_step(lse_mode=True)
    assert not r["mismatch"], r
    assert r["n_sel"] == [10, 60]


def test_all_keys_equal_uses_global_path():
    # constant logits: every candidate key is identical, the threshold digit holds
    # far more keys than the shared-memory stage keeps, ties resolve by flat index
    def flat(ls, t, x):
        return np.zeros_like(x)
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=64, vocab=4096, n_levels=2, codes_per_level=512,
                code_base=4096 - 1024, ctx_lens=[4], widths=[1024], n_items=[150000], seed=26)
    ls = LockStep(spec, logits_fn=flat)
    for t in range(2):
        r = ls.topk_step(lse_mode=True)
        assert not r["mismatch"], (t, r)


def test_row_without_candidates_turns_the_threshold_bound_off():
    """With at least W live rows the merge skips every key below the smallest row maximum (the
    rows' maxima are W candidates at or above it); a row without candidates has no maximum and
    must turn that bound off.  At level 1 every row gets one dominant valid code, so the rows'
    maxima are the only keys near the top.  One row's codes are NaN on the GPU (not candidates)
    and -inf for the oracle (candidates it never ranks among the first W here).  A bound taken
    over the other rows alone would leave only their W - 1 maxima and return W - 1 beams."""
    import torch
    from beam_decode_gb300 import binding as B
    W = 32
    spec = Spec(vocab=4096, n_levels=2, codes_per_level=64, code_base=4096 - 128, widths=[W],
                n_items=[3000], seed=27)
    ls = LockStep(spec)
    r = ls.topk_step(lse_mode=True)
    assert not r["mismatch"] and r["n_sel"] == [W], r
    ob = ls.obeams[0]
    x = ls.logits(1)
    lo = spec.code_base + spec.codes_per_level
    for b, pre in enumerate(ob.prefixes()):
        x[b, lo + ob.trie.valid_codes(pre)[0]] = 40.0
    dead = 5
    x_or, x_gpu = x.copy(), x.copy()
    x_or[dead, lo:lo + spec.codes_per_level] = -np.inf
    x_gpu[dead, lo:lo + spec.codes_per_level] = np.nan
    oinfo, lse32 = ls.oracle_topk(x_or)
    lse_in = torch.from_numpy(np.nan_to_num(lse32, nan=0.0)).cuda()
    ls.beam.constrained_topk(torch.from_numpy(x_gpu).cuda(), ld=x.shape[1], lse_in=lse_in)
    ls.beam.advance()
    assert ls.beam.status(clear=True) == B.GR_ERR_DEVICE  # the NaN keys are reported
    res = ls.compare_topk(oinfo, lse_mode=True)
    assert not res["mismatch"] and res["n_sel"] == [W], res


def test_minus_inf_and_huge_logits_outside_the_codes():
    """Logit rows holding -inf (banned tokens) in whole blocks, including the first values of
    each half a CTA reduces, and values of magnitude 1e30: the GPU's own log-sum-exp (no
    lse_in) stays within 1e-4 of the oracle's float64 one and the selection is the oracle's.
    The code logits stay ordinary, so every valid code keeps a finite log-probability."""
    def edit(ls, t, x):
        s = ls.spec
        x = x.copy()
        V = s.vocab
        x[:, :2048] = -np.inf
        x[:, V // 2:V // 2 + 1024] = -np.inf
        x[:, 4096:4160] = -1e30
        x[1::2, 2048:2052] = -np.inf
        return x
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=64, vocab=16384, n_levels=2, codes_per_level=256,
                code_base=16384 - 512, ctx_lens=[8, 8], widths=[64, 32], n_items=[20000, 20000], seed=28)
    ls = LockStep(spec, logits_fn=edit)
    for t in range(2):
        r = ls.topk_step(lse_mode=False)
        assert r["lse_err"] <= LP_TOL and r["lp_err"] <= LP_TOL, (t, r)
        assert not r["mismatch"], (t, r)


def test_many_requests_merge_in_smaller_clusters():
    """40 requests: their clusters of 8 merge CTAs would not fit the GPU at once (two per SM),
    so each request is merged by a cluster of 4; selections against the oracle, exact ties
    included (quantised logits), over two levels."""
    spec = Spec(vocab=2048, n_levels=3, codes_per_level=64, code_base=2048 - 192, ctx_lens=[8] * 40,
                widths=[48] * 40, n_items=[3000] * 40, seed=29)
    ls = LockStep(spec, logits_fn=lambda ls, t, x: np.round(x * 4.0) / 4.0)
    for t in range(3):
        r = ls.topk_step(lse_mode=True)
        assert not r["mismatch"], (t, r)

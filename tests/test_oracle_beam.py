"""Pins for the oracle's item-constrained beam search.

Semantics read from "Advancing Generative Recommendation Inference: our
collaboration with NVIDIA on TensorRT LLM" (section "Background: what
inference a recommendation request needs": keep the best prefixes, expand
and prune each step, return all surviving beams) and from the zhiding.cn
recsys-examples article (section "语义ID生成式推荐专用推理框架":
item-constrained top-K, dynamic beam width, BeamPath).

Pins: hand-worked fixtures (tests/golden), brute-force enumeration of every
item on tiny catalogues with prefix-keyed logits, a greedy walk for width 1,
argsort of the masked row for one level, and invariants.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from beam_decode_gb300.workload import draw_items
from oracle import OracleBeam, Trie, exhaustive_scores, log_softmax_row, token_id


def _prefix_logits(seed, V, std=2.0):
    cache = {}

    def f(prefix):
        key = tuple(prefix)
        if key not in cache:
            rng = np.random.default_rng([seed, len(key), *key])
            cache[key] = (rng.standard_normal(V) * std).astype(np.float32)
        return cache[key]
    return f


def _run(trie, width, L, C, base, logits_of_prefix, key_mode="f64"):
    ob = OracleBeam(trie, width, L, C, base, key_mode=key_mode)
    infos = []
    for _ in range(L):
        rows = np.stack([logits_of_prefix(p) for p in ob.prefixes()])
        infos.append(ob.step(rows))
    return ob, infos


# -- hand-worked fixtures --------------------------------------------------------

@pytest.mark.parametrize("name", ["hand_beam.json", "tie_across_beams.json"])
def test_golden_fixture(golden_dir, name):
    spec = json.load(open(os.path.join(golden_dir, name)))
    trie = Trie(np.array(spec["items"]), codes_per_level=spec["codes_per_level"])
    rows = {tuple(int(c) for c in k.split(",") if c != "") if k else (): np.log(np.array(w, dtype=np.float64))
            for k, w in spec["weights_by_prefix"].items()}
    for case in spec["cases"]:
        for mode in ("f64", "f32"):
            ob = OracleBeam(trie, case["width"], spec["n_levels"], spec["codes_per_level"], spec["code_base"],
                            key_mode=mode)
            tol = 1e-12 if mode == "f64" else 2e-6
            for lvl, key in enumerate(["expect_level0", "expect_final"]):
                ob.step(np.stack([rows[p] for p in ob.prefixes()]))
                exp = case[key]
                if lvl == 0:
                    assert ob.codes[0] == exp["codes"]
                else:
                    assert [list(p) for p in ob.prefixes()] == exp["codes"]
                assert ob.parents[lvl] == exp["parents"]
                for s, pr in zip(ob.scores[lvl], exp["probs"]):
                    assert abs(float(s) - np.log(float(Fraction(pr)))) < tol


# -- brute force ---------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_full_width_equals_exhaustive_ranking(seed):
    L, C, V, base = 2, 16, 1024, 512
    items = draw_items(50, L, C, "uniform", seed=seed)
    trie = Trie(items, codes_per_level=C)
    f = _prefix_logits(seed, V)
    width = max(trie.frontier_sizes())
    ob, _ = _run(trie, width, L, C, base, f)
    ex = exhaustive_scores(trie, f, base, C)
    got = ob.results()
    assert len(got) == len(ex) == 50
    ranked = sorted(ex.items(), key=lambda e: -e[1])
    assert [g[0] for g in got] == [r[0] for r in ranked]
    for g, r in zip(got, ranked):
        assert abs(g[2] - r[1]) < 1e-12


@pytest.mark.parametrize("seed,width", [(0, 1), (1, 3), (2, 4), (3, 7), (4, 16)])
def test_narrow_beam_scores_are_exhaustive_scores(seed, width):
    L, C, V, base = 3, 8, 256, 100
    items = draw_items(120, L, C, "uniform", seed=seed)
    trie = Trie(items, codes_per_level=C)
    f = _prefix_logits(seed + 10, V)
    ob, infos = _run(trie, width, L, C, base, f)
    ex = exhaustive_scores(trie, f, base, C)
    got = ob.results()
    assert len(got) == min(width, len(ex))
    for tup, iid, s in got:
        assert iid is not None and tup in ex
        assert abs(s - ex[tup]) < 1e-12
    scores = [g[2] for g in got]
    assert all(a >= b for a, b in zip(scores, scores[1:]))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_width_one_is_greedy_walk(seed):
    L, C, V, base = 3, 16, 512, 0
    items = draw_items(200, L, C, "zipf", seed=seed)
    trie = Trie(items, codes_per_level=C)
    f = _prefix_logits(seed, V)
    ob, _ = _run(trie, 1, L, C, base, f)
    # greedy: at each level the argmax of the log-probabilities over the valid codes
    prefix, total = (), 0.0
    for t in range(L):
        lp, _ = log_softmax_row(f(prefix))
        valid = trie.valid_codes(prefix)
        masked = np.full(C, -np.inf)
        masked[valid] = lp[base + t * C + np.array(valid)]
        c = int(np.argmax(masked))
        total += masked[c]
        prefix = prefix + (c,)
    (tup, iid, s), = ob.results()
    assert tup == prefix and abs(s - total) < 1e-12


def test_single_level_is_argsort_of_masked_row():
    C, V, base, W = 64, 300, 7, 10
    rng = np.random.default_rng(3)
    codes = rng.choice(C, size=25, replace=False)
    trie = Trie(codes[:, None], codes_per_level=C)
    x = (rng.standard_normal(V) * 2).astype(np.float32)
    x[base + codes[3]] = x[base + codes[4]]  # an exact tie
    ob = OracleBeam(trie, W, 1, C, base)
    ob.step(x[None])
    lp, _ = log_softmax_row(x)
    masked = np.full(C, -np.inf)
    masked[codes] = lp[base + codes]
    order = np.argsort(-masked, kind="stable")[:W]
    assert ob.codes[0] == [int(c) for c in order]


# -- invariants ------------------------------------------------------------------

@pytest.mark.parametrize("seed,width,dist", [(0, 8, "uniform"), (1, 32, "zipf"), (2, 5, "zipf")])
def test_invariants(seed, width, dist):
    L, C, V, base = 3, 16, 600, 40
    items = draw_items(300, L, C, dist, seed=seed)
    trie = Trie(items, codes_per_level=C)
    f = _prefix_logits(seed, V)
    ob = OracleBeam(trie, width, L, C, base)
    for t in range(L):
        prefixes = ob.prefixes()
        rows = np.stack([f(p) for p in prefixes])
        info = ob.step(rows)
        n_valid = sum(len(trie.valid_codes(p)) for p in prefixes)
        assert info["n_valid"] == n_valid
        assert len(ob.codes[t]) == min(width, n_valid)
        for i, (par, c) in enumerate(zip(ob.parents[t], ob.codes[t])):
            assert c in trie.valid_codes(prefixes[par])
        s = [float(v) for v in ob.scores[t]]
        assert all(a >= b for a, b in zip(s, s[1:]))
        if t > 0:  # a path's score never increases along the path (log-probs <= 0)
            prev = [float(v) for v in ob.scores[t - 1]]
            assert all(s[i] <= prev[ob.parents[t][i]] for i in range(len(s)))
    for tup, iid, sc in ob.results():
        assert trie.item(tup) == iid and iid is not None
        # parent chain reproduces the code string
    anc = ob.ancestry()
    for b, path in enumerate(anc):
        assert path[-1] == b
        for lvl in range(1, L):
            assert ob.parents[lvl][path[lvl]] == path[lvl - 1]


def test_f32_mode_keys_are_float32():
    L, C, V, base = 2, 16, 1024, 512
    items = draw_items(50, L, C, "uniform", seed=0)
    trie = Trie(items, codes_per_level=C)
    f = _prefix_logits(0, V)
    ob, infos = _run(trie, 4, L, C, base, f, key_mode="f32")
    for t in range(L):
        assert all(isinstance(s, np.float32) for s in ob.scores[t])
    ob64, _ = _run(trie, 4, L, C, base, f, key_mode="f64")
    for a, b in zip(ob.scores[-1], ob64.scores[-1]):
        assert abs(float(a) - b) < 1e-5


def test_trie_rejects_duplicates_and_out_of_range():
    with pytest.raises(ValueError):
        Trie(np.array([[0, 1], [0, 1]]))
    with pytest.raises(ValueError):
        Trie(np.array([[0, 16]]), codes_per_level=16)


def test_token_map():
    assert token_id(0, 0, 512, 16) == 512
    assert token_id(1, 15, 512, 16) == 543

"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, through monkeypatch)
-- a dropped term, a wrong sign, index or scale, a transposed operand, a
reversed tie-break -- and checks that at least one pin of
tests/test_oracle_*.py then fails.  Nothing here touches the CUDA path.
"""
import numpy as np
import pytest

import oracle.attention as oatt
import oracle.beam_search as obs
from tests import test_oracle_attention as T_att
from tests import test_oracle_beam as T_beam
from tests import test_oracle_logsoftmax as T_ls


def _fails(checks):
    for fn in checks:
        try:
            fn()
        except AssertionError:
            return True
    return False


def _attention_pins(golden_dir):
    return [
        lambda: T_att.test_matches_torch_sdpa(0, 4, 2, 16, 37, 5, 2),
        lambda: T_att.test_matches_torch_sdpa(2, 2, 1, 64, 64, 4, 3),
        T_att.test_equal_keys_give_mean_value,
        T_att.test_single_key_gives_its_value,
        T_att.test_two_keys_scale_closed_form,
        T_att.test_gqa_head_mapping,
        T_att.test_ancestry_selects_path_slots,
        T_att.test_lse_split_identity,
    ]


def _beam_pins(golden_dir):
    return [
        lambda: T_beam.test_golden_fixture(golden_dir, "hand_beam.json"),
        lambda: T_beam.test_golden_fixture(golden_dir, "tie_across_beams.json"),
        lambda: T_beam.test_full_width_equals_exhaustive_ranking(0),
        lambda: T_beam.test_narrow_beam_scores_are_exhaustive_scores(1, 3),
        lambda: T_beam.test_width_one_is_greedy_walk(0),
        T_beam.test_single_level_is_argsort_of_masked_row,
        lambda: T_beam.test_invariants(0, 8, "uniform"),
        lambda: T_ls.test_matches_scipy_and_torch(0, 0.0, 2.0),
        T_ls.test_normalised_and_shift_invariant,
        T_ls.test_uniform_row_closed_form,
    ]


# -- attention mutations -----------------------------------------------------------

def _attend_scale_1_over_d(q, keys, values, scale):
    d = len(q)
    return _orig_attend(q, keys, values, 1.0 / d)


def _attend_no_scale(q, keys, values, scale):
    return _orig_attend(q, keys, values, 1.0)


def _attend_transposed(q, keys, values, scale):
    q = np.asarray(q, dtype=np.float64)
    s = (np.asarray(keys, dtype=np.float64) @ q) * scale
    p = np.exp(s - s.max())
    v = np.asarray(values, dtype=np.float64)
    n, d = v.shape
    vt = v.T.reshape(n, d) if n == d else v[::-1]
    return (p @ vt) / p.sum(), float(s.max() + np.log(p.sum()))


def _attend_unnormalised(q, keys, values, scale):
    q = np.asarray(q, dtype=np.float64)
    s = (np.asarray(keys, dtype=np.float64) @ q) * scale
    p = np.exp(s - s.max())
    return p @ np.asarray(values, dtype=np.float64), float(s.max() + np.log(p.sum()))


def _attend_drop_last_key(q, keys, values, scale):
    keys = np.asarray(keys)
    values = np.asarray(values)
    if len(keys) > 1:
        keys, values = keys[:-1], values[:-1]
    return _orig_attend(q, keys, values, scale)


_orig_attend = oatt.attend_row


def _beam_attention_gqa_mod(q, ctx_k, ctx_v, beam_k, beam_v, ancestry, beams=None):
    # query head q reads KV head q % Hkv instead of q // G
    q = np.asarray(q, dtype=np.float64)
    hq, d = q.shape[1], q.shape[2]
    hkv = ctx_k.shape[0]
    out = np.zeros((q.shape[0], hq, d))
    for b in range(q.shape[0]):
        for h in range(hq):
            kv = h % hkv
            keys = np.concatenate([ctx_k[kv]] + [beam_k[j][s, kv][None] for j, s in enumerate(ancestry[b])])
            vals = np.concatenate([ctx_v[kv]] + [beam_v[j][s, kv][None] for j, s in enumerate(ancestry[b])])
            out[b, h], _ = _orig_attend(q[b, h], keys, vals, 1 / np.sqrt(d))
    return out


def _beam_attention_reversed_path(q, ctx_k, ctx_v, beam_k, beam_v, ancestry, beams=None):
    return _orig_beam_attention(q, ctx_k, ctx_v, beam_k, beam_v, [list(a)[::-1] for a in ancestry], beams)


def _beam_attention_no_beam_keys(q, ctx_k, ctx_v, beam_k, beam_v, ancestry, beams=None):
    return _orig_beam_attention(q, ctx_k, ctx_v, beam_k, beam_v, [[] for _ in ancestry], beams)


_orig_beam_attention = oatt.beam_attention


@pytest.mark.parametrize("name,target,fn", [
    ("scale 1/D", "attend_row", _attend_scale_1_over_d),
    ("no scale", "attend_row", _attend_no_scale),
    ("values transposed/reversed", "attend_row", _attend_transposed),
    ("no normalisation", "attend_row", _attend_unnormalised),
    ("last key dropped", "attend_row", _attend_drop_last_key),
    ("gqa q % Hkv", "beam_attention", _beam_attention_gqa_mod),
    ("ancestry reversed", "beam_attention", _beam_attention_reversed_path),
    ("beam keys dropped", "beam_attention", _beam_attention_no_beam_keys),
])
def test_attention_mutation_is_caught(monkeypatch, golden_dir, name, target, fn):
    monkeypatch.setattr(oatt, target, fn)
    monkeypatch.setattr(T_att, target, fn)  # beam_attention reaches attend_row through its module
    assert _fails(_attention_pins(golden_dir)), name


# -- beam search mutations ---------------------------------------------------------

_orig_ls = obs.log_softmax_row
_orig_rank = obs.rank_candidates
_orig_token = obs.token_id


def _ls_sign(x):
    lp, lse = _orig_ls(x)
    return -lp, lse


def _ls_drop_lse(x):
    x = np.asarray(x, dtype=np.float64)
    return x - x.max(), float(x.max())


def _rank_tie_desc(c):
    return sorted(c, key=lambda e: (-float(e[0]), -e[1]))


def _rank_ascending(c):
    return sorted(c, key=lambda e: (float(e[0]), e[1]))


def _rank_by_code(c):
    return sorted(c, key=lambda e: (-float(e[0]), e[3], e[2]))


def _token_off_by_one(level, code, base, C):
    return base + level * C + code + 1


def _token_level_swapped(level, code, base, C):
    return base + code * C + level if code * C + level < 2 * C else base + level * C + code


class _RenormBeam(obs.OracleBeam):
    """Renormalises log-probabilities over the valid codes (reading 1 violated)."""

    def step(self, logits, lse_in=None):
        t = self.t
        rows = []
        lo = obs.token_id(t, 0, self.code_base, self.C)
        for b, pre in enumerate(self.prefixes()):
            r = np.full(np.shape(logits[b]), -1e30)
            valid = lo + np.array(self.trie.valid_codes(pre))
            r[valid] = np.asarray(logits[b], dtype=np.float64)[valid]
            rows.append(r)
        return super().step(np.stack(rows), lse_in)


class _NoScoreBeam(obs.OracleBeam):
    """Forgets the parent's score (dropped term S_b)."""

    def beam_scores(self):
        return [0.0] * self.n_live()


@pytest.mark.parametrize("name,target,fn", [
    ("log-softmax sign flipped", "log_softmax_row", _ls_sign),
    ("log-softmax drops lse", "log_softmax_row", _ls_drop_lse),
    ("tie-break flat descending", "rank_candidates", _rank_tie_desc),
    ("ascending sort", "rank_candidates", _rank_ascending),
    ("tie-break by code first", "rank_candidates", _rank_by_code),
    ("token map off by one", "token_id", _token_off_by_one),
    ("token map level/code swapped", "token_id", _token_level_swapped),
])
def test_beam_mutation_is_caught(monkeypatch, golden_dir, name, target, fn):
    monkeypatch.setattr(obs, target, fn)
    assert _fails(_beam_pins(golden_dir)), name


@pytest.mark.parametrize("cls", [_RenormBeam, _NoScoreBeam])
def test_beam_class_mutation_is_caught(monkeypatch, golden_dir, cls):
    monkeypatch.setattr(T_beam, "OracleBeam", cls)
    assert _fails(_beam_pins(golden_dir)), cls.__name__


# -- float32 key mutations ---------------------------------------------------------

def _key_one_rounding(score32, x32, lse32):
    # the exact S + x - LSE (float64 is exact at these magnitudes) rounded once
    return np.float32(float(score32) + (float(x32) - float(lse32)))


def _key_other_association(score32, x32, lse32):
    return np.float32(np.float32(np.float32(score32) + np.float32(x32)) - np.float32(lse32))


def _key_drops_score(score32, x32, lse32):
    return np.float32(np.float32(x32) - np.float32(lse32))


def _key_pins(golden_dir):
    return [T_ls.test_key_f32_is_two_roundings_of_exact_values] + _beam_pins(golden_dir)


@pytest.mark.parametrize("name,fn", [
    ("key rounded once", _key_one_rounding),
    ("key summed in the other order", _key_other_association),
    ("key without the beam score", _key_drops_score),
])
def test_key_f32_mutation_is_caught(monkeypatch, golden_dir, name, fn):
    monkeypatch.setattr(obs, "key_f32", fn)
    assert _fails(_key_pins(golden_dir)), name


# -- multi-item scoring mutations ---------------------------------------------------

import oracle.scoring as osc
from tests import test_oracle_scoring as T_sc

_orig_mia = osc.multi_item_attention
_orig_labels = osc.label_logprobs
_orig_srank = osc.rank


def _scoring_pins():
    return [
        lambda: T_sc.test_matches_sdpa_on_the_joined_sequence(0, 4, 2, 16, 23, (3, 1, 4, 2)),
        lambda: T_sc.test_matches_sdpa_on_the_joined_sequence(3, 8, 2, 32, 70, (16, 2, 9)),
        T_sc.test_other_candidates_and_later_tokens_are_invisible,
        T_sc.test_equal_keys_give_mean_value,
        T_sc.test_label_logprobs_match_scipy,
        T_sc.test_rank_orders_by_score_then_index,
    ]


def _mia_whole_segment(q, pk, pv, sk, sv, seg_lens, rows=None):
    # every token of a candidate sees the candidate's later tokens too (no causality)
    hq, d = q.shape[1], q.shape[2]
    g = hq // pk.shape[0]
    cand, _ = osc.segment_rows(seg_lens)
    rows = range(q.shape[0]) if rows is None else rows
    out = np.zeros((len(rows), hq, d))
    for i, r in enumerate(rows):
        own = np.where(cand == cand[r])[0]
        for h in range(hq):
            keys = np.concatenate([pk[h // g], sk[own, h // g]])
            vals = np.concatenate([pv[h // g], sv[own, h // g]])
            out[i, h], _ = oatt.attend_row(q[r, h], keys, vals, 1 / np.sqrt(d))
    return out


def _mia_sees_previous_candidate(q, pk, pv, sk, sv, seg_lens, rows=None):
    # the mask leaks the previous candidate's tokens (a plain causal mask over the joined sequence)
    hq, d = q.shape[1], q.shape[2]
    g = hq // pk.shape[0]
    rows = range(q.shape[0]) if rows is None else rows
    out = np.zeros((len(rows), hq, d))
    for i, r in enumerate(rows):
        for h in range(hq):
            keys = np.concatenate([pk[h // g], sk[:r + 1, h // g]])
            vals = np.concatenate([pv[h // g], sv[:r + 1, h // g]])
            out[i, h], _ = oatt.attend_row(q[r, h], keys, vals, 1 / np.sqrt(d))
    return out


def _mia_no_prefix(q, pk, pv, sk, sv, seg_lens, rows=None):
    return _orig_mia(q, pk[:, :0], pv[:, :0], sk, sv, seg_lens, rows)


def _labels_off_by_one(logits, label_ids):
    V = np.asarray(logits).shape[1]
    return _orig_labels(logits, [(l + 1) % V for l in label_ids])


def _labels_raw_logits(logits, label_ids):
    return np.asarray(logits, dtype=np.float64)[:, list(label_ids)]


def _rank_ties_high_index(scores):
    s = list(scores)
    return np.array(sorted(range(len(s)), key=lambda c: (-s[c], -c)), dtype=np.int32)


@pytest.mark.parametrize("name,target,fn", [
    ("segment not causal", "multi_item_attention", _mia_whole_segment),
    ("previous candidate visible", "multi_item_attention", _mia_sees_previous_candidate),
    ("prefix dropped", "multi_item_attention", _mia_no_prefix),
    ("label index off by one", "label_logprobs", _labels_off_by_one),
    ("labels not normalised", "label_logprobs", _labels_raw_logits),
    ("ties by higher index", "rank", _rank_ties_high_index),
])
def test_scoring_mutation_is_caught(monkeypatch, name, target, fn):
    monkeypatch.setattr(osc, target, fn)
    monkeypatch.setattr(T_sc, target, fn)
    assert _fails(_scoring_pins()), name

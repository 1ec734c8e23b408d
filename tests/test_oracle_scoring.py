"""Pins for the oracle's multi-item scoring.

"Advancing Generative Recommendation Inference: our collaboration with NVIDIA
on TensorRT LLM", sections "Background: what inference a recommendation
request needs" and "Scoring many candidates at once": user prefix and all
candidates in one sequence, a mask that lets each candidate see only the
prefix and itself, label-token log-probabilities read out, candidates ranked
by them.  Pins: a library routine (torch scaled_dot_product_attention in
float64 on the whole joined sequence with an explicit boolean mask), the
isolation and causality the mask implies, a closed form, scipy's
log_softmax, and a hand-checked ranking with ties.
"""
import numpy as np
import pytest
import torch
from scipy.special import log_softmax

from oracle.scoring import label_logprobs, multi_item_attention, rank, segment_rows


def _case(seed, hq=4, hkv=2, d=16, T=23, seg_lens=(3, 1, 4, 2)):
    rng = np.random.default_rng(seed)
    R = int(sum(seg_lens))
    q = rng.standard_normal((R, hq, d))
    pk, pv = rng.standard_normal((hkv, T, d)), rng.standard_normal((hkv, T, d))
    sk, sv = rng.standard_normal((R, hkv, d)), rng.standard_normal((R, hkv, d))
    return q, pk, pv, sk, sv, list(seg_lens)


def _sdpa_joined(q, pk, pv, sk, sv, seg_lens):
    """The whole joined sequence [prefix; cand_0; cand_1; ...] through torch SDPA with the
    multi-item mask written out position by position."""
    hq, d = q.shape[1], q.shape[2]
    hkv, T = pk.shape[0], pk.shape[1]
    R = q.shape[0]
    keys = np.concatenate([pk, sk.transpose(1, 0, 2)], axis=1)      # [Hkv, T + R, D]
    vals = np.concatenate([pv, sv.transpose(1, 0, 2)], axis=1)
    owner = np.repeat(np.arange(len(seg_lens)), seg_lens)          # candidate of each row
    mask = np.zeros((R, T + R), dtype=bool)
    for i in range(R):
        mask[i, :T] = True                                           # the whole user prefix
        for j in range(R):
            mask[i, T + j] = owner[j] == owner[i] and j <= i          # itself, causally
    g = hq // hkv
    k = torch.from_numpy(np.repeat(keys, g, axis=0))                  # [Hq, T + R, D]
    v = torch.from_numpy(np.repeat(vals, g, axis=0))
    qq = torch.from_numpy(q.transpose(1, 0, 2).copy())                # [Hq, R, D]
    out = torch.nn.functional.scaled_dot_product_attention(qq, k, v, attn_mask=torch.from_numpy(mask))
    return out.numpy().transpose(1, 0, 2)


@pytest.mark.parametrize("seed,hq,hkv,d,T,seg", [(0, 4, 2, 16, 23, (3, 1, 4, 2)), (1, 16, 8, 128, 40, (5, 5)),
                                                 (2, 2, 1, 64, 1, (1, 1, 1)), (3, 8, 2, 32, 70, (16, 2, 9))])
def test_matches_sdpa_on_the_joined_sequence(seed, hq, hkv, d, T, seg):
    q, pk, pv, sk, sv, sl = _case(seed, hq, hkv, d, T, seg)
    got = multi_item_attention(q, pk, pv, sk, sv, sl)
    np.testing.assert_allclose(got, _sdpa_joined(q, pk, pv, sk, sv, sl), rtol=1e-12, atol=1e-12)


def test_other_candidates_and_later_tokens_are_invisible():
    q, pk, pv, sk, sv, sl = _case(4)
    base = multi_item_attention(q, pk, pv, sk, sv, sl)
    cand, pos = segment_rows(sl)
    # change candidate 2 entirely: rows of the other candidates do not move
    sk2, sv2 = sk.copy(), sv.copy()
    sk2[cand == 2] += 3.0
    sv2[cand == 2] -= 2.0
    moved = multi_item_attention(q, pk, pv, sk2, sv2, sl)
    np.testing.assert_array_equal(moved[cand != 2], base[cand != 2])
    assert not np.allclose(moved[cand == 2], base[cand == 2])
    # change the last token of candidate 0: its earlier rows do not move, its last row does
    last0 = int(np.where(cand == 0)[0][-1])
    sk3 = sk.copy()
    sk3[last0] += 5.0
    m3 = multi_item_attention(q, pk, pv, sk3, sv, sl)
    np.testing.assert_array_equal(m3[:last0], base[:last0])
    assert not np.allclose(m3[last0], base[last0])


def test_equal_keys_give_mean_value():
    hkv, d, T, sl = 1, 8, 5, [2, 3]
    R = sum(sl)
    q = np.random.default_rng(5).standard_normal((R, 2, d))
    pk = np.ones((hkv, T, d))
    sk = np.ones((R, hkv, d))
    pv = np.arange(T * d, dtype=np.float64).reshape(hkv, T, d)
    sv = 100.0 + np.arange(R * d, dtype=np.float64).reshape(R, hkv, d)
    out = multi_item_attention(q, pk, pv, sk, sv, sl)
    # row 3 = candidate 1, position 1: sees the 5 prefix values and rows 2, 3
    exp = (pv[0].sum(axis=0) + sv[2, 0] + sv[3, 0]) / (T + 2)
    np.testing.assert_allclose(out[3, 0], exp, rtol=1e-13)
    np.testing.assert_allclose(out[3, 1], exp, rtol=1e-13)


def test_label_logprobs_match_scipy():
    x = np.random.default_rng(6).standard_normal((7, 301)) * 2.0
    labels = [5, 300, 0, 17]
    np.testing.assert_allclose(label_logprobs(x, labels), log_softmax(x, axis=1)[:, labels], rtol=1e-13, atol=1e-13)


def test_rank_orders_by_score_then_index():
    # hand-checked: 0.5 (c2) > 0.1 (c0 = c3, tie -> lower index first) > -1 (c1) > -2 (c4)
    assert rank([0.1, -1.0, 0.5, 0.1, -2.0]).tolist() == [2, 0, 3, 1, 4]

"""Pins for the oracle's naive per-beam attention.

zhiding.cn recsys-examples article, section "语义ID生成式推荐专用推理框架":
each beam attends to the shared request context (ContextKV) followed by the
tokens of its own path (BeamKV, found through BeamPath).  Pins: a library
routine (torch scaled_dot_product_attention in float64 on the concatenated
sequence), closed forms, the GQA head mapping, the ancestry indexing, the
1/sqrt(D) scale, and the log-sum-exp split identity.
"""
import numpy as np
import pytest
import torch

from oracle import attend_row, beam_attention


def _rand_case(seed, hq=4, hkv=2, d=16, T=37, W=5, t=2):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((W, hq, d))
    ck = rng.standard_normal((hkv, T, d))
    cv = rng.standard_normal((hkv, T, d))
    bk = [rng.standard_normal((W, hkv, d)) for _ in range(t)]
    bv = [rng.standard_normal((W, hkv, d)) for _ in range(t)]
    anc = [[int(rng.integers(0, W)) for _ in range(t - 1)] + [b] for b in range(W)]
    return q, ck, cv, bk, bv, anc


@pytest.mark.parametrize("seed,hq,hkv,d,T,W,t", [(0, 4, 2, 16, 37, 5, 2), (1, 16, 8, 128, 130, 3, 1),
                                                 (2, 2, 1, 64, 64, 4, 3), (3, 8, 1, 32, 1, 2, 2)])
def test_matches_torch_sdpa(seed, hq, hkv, d, T, W, t):
    q, ck, cv, bk, bv, anc = _rand_case(seed, hq, hkv, d, T, W, t)
    out = beam_attention(q, ck, cv, bk, bv, anc)
    g = hq // hkv
    for b in range(W):
        for h in range(hq):
            kv = h // g
            keys = np.concatenate([ck[kv]] + [bk[j][anc[b][j], kv][None] for j in range(t)])
            vals = np.concatenate([cv[kv]] + [bv[j][anc[b][j], kv][None] for j in range(t)])
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[b, h][None, None, None]), torch.from_numpy(keys[None, None]),
                torch.from_numpy(vals[None, None]))[0, 0, 0].numpy()
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-12)


def test_equal_keys_give_mean_value():
    rng = np.random.default_rng(7)
    k = np.tile(rng.standard_normal(32), (50, 1))
    v = rng.standard_normal((50, 32))
    o, lse = attend_row(rng.standard_normal(32), k, v, 0.3)
    np.testing.assert_allclose(o, v.mean(axis=0), atol=1e-13)


def test_single_key_gives_its_value():
    rng = np.random.default_rng(8)
    v = rng.standard_normal((1, 8))
    o, lse = attend_row(rng.standard_normal(8), rng.standard_normal((1, 8)), v, 1.0)
    np.testing.assert_allclose(o, v[0], atol=0)


def test_two_keys_scale_closed_form():
    d = 64
    q = np.zeros(d); q[0] = 1.0
    k = np.zeros((2, d)); k[0, 0] = 8.0; k[1, 0] = 0.0
    v = np.array([[1.0] + [0] * (d - 1), [0.0] * d])
    o, lse = attend_row(q, k, v, 1.0 / np.sqrt(d))
    # scores 8/8 = 1 and 0 -> weight of key 0 is e/(1+e)
    assert abs(o[0] - np.e / (1 + np.e)) < 1e-15
    assert abs(lse - np.log(1 + np.e)) < 1e-15


def test_gqa_head_mapping():
    # KV head h holds value h everywhere: query head q must read KV head q // G
    W, hq, hkv, d, T = 2, 8, 4, 8, 5
    rng = np.random.default_rng(9)
    q = rng.standard_normal((W, hq, d))
    ck = rng.standard_normal((hkv, T, d))
    cv = np.stack([np.full((T, d), float(h)) for h in range(hkv)])
    bk = [rng.standard_normal((W, hkv, d))]
    bv = [np.broadcast_to(np.arange(hkv, dtype=np.float64)[None, :, None], (W, hkv, d)).copy()]
    out = beam_attention(q, ck, cv, bk, bv, [[0], [1]])
    for h in range(hq):
        np.testing.assert_allclose(out[:, h], h // (hq // hkv), atol=1e-12)


def test_ancestry_selects_path_slots():
    # context keys score 0, beam keys are large along q: each beam's output is
    # dominated by the values at its own ancestors' slots
    W, d, T, t = 4, 8, 3, 2
    q = np.zeros((W, 1, d)); q[:, 0, 0] = 1.0
    ck = np.zeros((1, T, d)); cv = np.zeros((1, T, d))
    bk = [np.zeros((W, 1, d)) for _ in range(t)]
    bv = [np.zeros((W, 1, d)) for _ in range(t)]
    for j in range(t):
        for s in range(W):
            bk[j][s, 0, 0] = 200.0
            bv[j][s, 0, :] = 10 * j + s
    anc = [[3, 0], [1, 1], [0, 2], [2, 3]]
    out = beam_attention(q, ck, cv, bk, bv, anc)
    for b in range(W):
        expect = 0.5 * ((10 * 0 + anc[b][0]) + (10 * 1 + anc[b][1]))
        np.testing.assert_allclose(out[b, 0, 0], expect, atol=1e-9)


def test_lse_split_identity():
    # attention over [A; B] equals the log-sum-exp weighted mix of the parts
    rng = np.random.default_rng(11)
    q = rng.standard_normal(16)
    ka, va = rng.standard_normal((40, 16)), rng.standard_normal((40, 16))
    kb, vb = rng.standard_normal((3, 16)), rng.standard_normal((3, 16))
    sc = 0.25
    o, l = attend_row(q, np.concatenate([ka, kb]), np.concatenate([va, vb]), sc)
    oa, la = attend_row(q, ka, va, sc)
    ob, lb = attend_row(q, kb, vb, sc)
    lt = np.logaddexp(la, lb)
    np.testing.assert_allclose(o, np.exp(la - lt) * oa + np.exp(lb - lt) * ob, atol=1e-13)
    assert abs(l - lt) < 1e-13

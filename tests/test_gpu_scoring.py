"""Multi-item candidate scoring through the C ABI against the CPU oracle.

"Advancing Generative Recommendation Inference: our collaboration with NVIDIA
on TensorRT LLM", sections "Background: what inference a recommendation
request needs" and "Scoring many candidates at once": each candidate token
attends to the user prefix and to its own candidate up to itself; label-token
log-probabilities at each candidate's last token rank the candidates.
"""
import numpy as np
import pytest

from beam_decode_gb300 import binding as B
from beam_decode_gb300 import workload as wl
from oracle.scoring import label_logprobs, multi_item_attention, rank
from tests.harness import ATOL, LP_TOL, RTOL

pytestmark = pytest.mark.gpu


def _setup(seed, n_layers, hq, hkv, d, vocab, prefixes, segs, labels):
    import torch
    off, offs = 4, []
    for T in prefixes:
        offs.append(off)
        off += T + 11
    ck = wl.round_to_bf16(wl.host_normal((n_layers, hkv, off, d), seed, wl.TAG_CTX_K))
    cv = wl.round_to_bf16(wl.host_normal((n_layers, hkv, off, d), seed, wl.TAG_CTX_V))
    sc = B.Score(n_layers, hq, hkv, d, vocab, labels, torch.from_numpy(ck).to(torch.bfloat16).cuda(),
                 torch.from_numpy(cv).to(torch.bfloat16).cuda(),
                 [(offs[r], prefixes[r], segs[r]) for r in range(len(prefixes))])
    rows = sc.rows
    sk = wl.round_to_bf16(wl.host_normal((n_layers, rows, hkv, d), seed, wl.TAG_BEAM_K))
    sv = wl.round_to_bf16(wl.host_normal((n_layers, rows, hkv, d), seed, wl.TAG_BEAM_V))
    sc.seg_k.copy_(torch.from_numpy(sk).to(torch.bfloat16))
    sc.seg_v.copy_(torch.from_numpy(sv).to(torch.bfloat16))
    return sc, ck, cv, sk, sv, offs


def _check_attention(sc, ck, cv, sk, sv, offs, prefixes, segs, layer, seed, sample=None):
    import torch
    hq, d = sc.cfg.n_q_heads, sc.cfg.head_dim
    q = wl.round_to_bf16(wl.host_normal((sc.rows, hq, d), seed, wl.TAG_Q, sub=(layer,)))
    gq = torch.from_numpy(q).to(torch.bfloat16).cuda()
    out = torch.full_like(gq, float("nan"))
    sc.attn(layer, gq, out)
    got = out.float().cpu().numpy()
    worst = 0.0
    for r, (T, seg) in enumerate(zip(prefixes, segs)):
        r0, r1 = sc.row_offsets[r], sc.row_offsets[r + 1]
        rows = list(range(r1 - r0)) if sample is None else sorted(set(min(x, r1 - r0 - 1) for x in sample))
        ref = multi_item_attention(q[r0:r1], ck[layer, :, offs[r]:offs[r] + T], cv[layer, :, offs[r]:offs[r] + T],
                                   sk[layer, r0:r1], sv[layer, r0:r1], seg, rows=rows)
        g = got[r0 + np.array(rows)]
        assert not np.isnan(g).any()
        worst = max(worst, float(np.max(np.abs(g - ref) / (ATOL + RTOL * np.abs(ref)))))
    return worst


def _check_labels(sc, vocab, labels, seed):
    import torch
    x = wl.host_normal((sc.n_candidates, vocab), seed, wl.TAG_LOGITS, std=2.0)
    lp, rk = sc.labels(torch.from_numpy(x).cuda())
    lp, rk = lp.cpu().numpy(), rk.cpu().numpy()
    ref = label_logprobs(x, labels)
    assert np.max(np.abs(lp - ref)) <= LP_TOL
    # the ranking is unique given the GPU's fp32 log-probabilities: it must be exactly their order
    for r in range(sc.n_requests):
        c0, c1 = sc.cand_offsets[r], sc.cand_offsets[r + 1]
        assert np.array_equal(rk[c0:c1], rank(lp[c0:c1, 0].astype(np.float64)))
        # and agree with the oracle's order wherever the oracle's scores are not within tolerance
        exp = rank(ref[c0:c1, 0])
        gap = np.abs(np.diff(ref[c0:c1, 0][exp]))
        mine = rk[c0:c1]
        for i in np.where(gap > 2 * LP_TOL)[0]:  # a clear gap after position i: same top i+1
            assert set(mine[:i + 1].tolist()) == set(exp[:i + 1].tolist())


def test_scoring_ragged_segments_two_requests():
    rng = np.random.default_rng(7)
    segs = [list(rng.integers(1, 17, size=60)), [1, 16, 3, 9, 2]]
    prefixes = [300, 1]
    labels = [7, 2047, 0]
    sc, ck, cv, sk, sv, offs = _setup(70, 2, 4, 2, 64, 2048, prefixes, segs, labels)
    for layer in range(2):
        assert _check_attention(sc, ck, cv, sk, sv, offs, prefixes, segs, layer, 70) <= 1.0
    _check_labels(sc, 2048, labels, 70)
    assert sc.status() == 0


def test_scoring_qwen_geometry_500_candidates():
    # the pages' scoring call: 500 candidates per request; Qwen3-1.7B attention geometry
    rng = np.random.default_rng(8)
    segs = [list(rng.integers(4, 13, size=500))]
    prefixes = [2000]
    labels = [9454, 2753]
    sc, ck, cv, sk, sv, offs = _setup(71, 1, 16, 8, 128, 151936, prefixes, segs, labels)
    sample = list(range(0, sc.rows, 97)) + [sc.rows - 1]
    assert _check_attention(sc, ck, cv, sk, sv, offs, prefixes, segs, 0, 71, sample=sample) <= 1.0
    _check_labels(sc, 151936, labels, 71)
    assert sc.status() == 0


def test_scoring_many_one_token_candidates():
    # 1024 candidates of one token (the ranking's maximum) with a short prefix
    segs = [[1] * 1024]
    prefixes = [129]
    labels = [5]
    sc, ck, cv, sk, sv, offs = _setup(72, 1, 2, 1, 64, 1024, prefixes, segs, labels)
    assert _check_attention(sc, ck, cv, sk, sv, offs, prefixes, segs, 0, 72) <= 1.0
    _check_labels(sc, 1024, labels, 72)
    assert sc.status() == 0


def test_scoring_rejects_bad_requests():
    import torch
    ck = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.GrError) as e:
        B.Score(1, 2, 1, 64, 1024, [5], ck, ck, [(0, 10, [17])])
    assert e.value.status == B.GR_ERR_CAPACITY
    with pytest.raises(B.GrError) as e:
        B.Score(1, 2, 1, 64, 1024, [1024], ck, ck, [(0, 10, [3])])
    assert e.value.status == B.GR_ERR_INVALID_ARG
    with pytest.raises(B.GrError) as e:
        B.Score(1, 2, 1, 64, 1024, [5], ck, ck, [(60, 10, [3])])
    assert e.value.status == B.GR_ERR_INVALID_ARG

"""Multi-item candidate scoring, computed naively (oracle, test infrastructure).

[GRINF] "Advancing Generative Recommendation Inference: our collaboration with
NVIDIA on TensorRT LLM", English page:
  * section "Background: what inference a recommendation request needs":
    existing candidates are put into the prompt, the model's log-probabilities
    of label tokens such as "yes" / "no" are read out, and the candidates are
    ranked by them;
  * section "Scoring many candidates at once": multi-item scoring joins the
    user prefix and all candidates into one sequence, and an attention mask
    lets each candidate see only the user prefix and itself, so one forward
    pass scores every candidate.

Readings where the pages are silent:
  * inside its own segment a candidate token sees the candidate's tokens up to
    and including itself (causal, as in any decoder forward pass); it sees the
    whole user prefix and no other candidate;
  * the label log-probabilities of a candidate are read at its last token:
    log-softmax over the full vocabulary, then the label tokens' entries;
  * the ranking orders candidates by the first label's log-probability,
    highest first, ties by candidate index;
  * as in the decode oracle: grouped-query heads (q reads KV head q // G),
    scale 1/sqrt(D), float64 arithmetic on the stored values.

The fast path keeps the user prefix as a shared context read once per request
and each candidate's own tokens as private keys; the oracle builds every
row's visible sequence explicitly.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from .attention import attend_row
from .beam_search import log_softmax_row


def segment_rows(seg_lens: Sequence[int]):
    """Row layout of the candidates' tokens: for each row, (candidate, position)."""
    cand, pos = [], []
    for c, n in enumerate(seg_lens):
        for p in range(int(n)):
            cand.append(c)
            pos.append(p)
    return np.array(cand, dtype=np.int64), np.array(pos, dtype=np.int64)


def multi_item_attention(q: np.ndarray, prefix_k: np.ndarray, prefix_v: np.ndarray,
                         seg_k: np.ndarray, seg_v: np.ndarray, seg_lens: Sequence[int],
                         rows: Sequence[int] = None) -> np.ndarray:
    """Attention output of candidate-token rows under the multi-item mask.

    q          [R, Hq, D]    one row per candidate token, candidates in order
    prefix_k/v [Hkv, T, D]   the user prefix's keys / values
    seg_k/v    [R, Hkv, D]   keys / values of the candidate tokens, same rows as q
    seg_lens   tokens of each candidate (sum = R)
    rows       rows to evaluate (default: all)

    Returns float64 [len(rows), Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    n_q_heads, d = q.shape[1], q.shape[2]
    group = n_q_heads // prefix_k.shape[0]
    scale = 1.0 / np.sqrt(d)
    cand, pos = segment_rows(seg_lens)
    first = np.concatenate([[0], np.cumsum(seg_lens)[:-1]]).astype(np.int64)
    if rows is None:
        rows = range(q.shape[0])
    out = np.zeros((len(rows), n_q_heads, d), dtype=np.float64)
    for i, r in enumerate(rows):
        own = range(first[cand[r]], first[cand[r]] + pos[r] + 1)  # its candidate's tokens up to itself
        for qh in range(n_q_heads):
            kvh = qh // group
            keys = np.concatenate([prefix_k[kvh], np.asarray(seg_k)[list(own), kvh]], axis=0)
            values = np.concatenate([prefix_v[kvh], np.asarray(seg_v)[list(own), kvh]], axis=0)
            out[i, qh], _ = attend_row(q[r, qh], keys, values, scale)
    return out


def label_logprobs(logits: np.ndarray, label_ids: Sequence[int]) -> np.ndarray:
    """Full-vocabulary log-probabilities of the label tokens, one row per candidate
    (the logits of its last token): float64 [n_cand, n_labels]."""
    out = np.zeros((logits.shape[0], len(label_ids)), dtype=np.float64)
    for c in range(logits.shape[0]):
        lp, _ = log_softmax_row(logits[c])
        out[c] = lp[list(label_ids)]
    return out


def rank(scores: Sequence[float]) -> np.ndarray:
    """Candidate indices by score, highest first, ties by index."""
    s = list(scores)
    return np.array(sorted(range(len(s)), key=lambda c: (-s[c], c)), dtype=np.int32)

"""Decode attention of every beam, computed naively (oracle, test infrastructure).

[RECSYS] section "语义ID生成式推荐专用推理框架": the long request context is
kept once per request (ContextKV), each beam keeps the short history of its
own decoded tokens (BeamKV), and beam ancestry is tracked (BeamPath), so that
a beam is not stored as an independent long sequence.  What a beam attends
to is still its whole sequence: the request's context followed by the tokens
on its own path.  The oracle therefore builds, for each beam, that
concatenated sequence explicitly and runs textbook softmax attention over
it -- the layout savings are the fast path's business, not the oracle's.

Readings where the pages are silent:
  * grouped-query attention: query head q reads KV head q // G, G = Hq / Hkv
    (the Qwen3 convention of repeating each KV head over G consecutive query
    heads);
  * scale 1 / sqrt(head_dim); no mask inside the context (a decode token sees
    the whole history); Q and K arrive already position-encoded;
  * arithmetic in float64 on the stored (bf16-representable) values.
"""
from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np


def attend_row(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float
               ) -> Tuple[np.ndarray, float]:
    """softmax(scale * keys @ q) @ values for one query row, in float64.

    Returns (output [D], natural-log log-sum-exp of the scaled scores).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    s = (keys @ q) * scale
    m = s.max()
    p = np.exp(s - m)
    z = p.sum()
    return (p @ values) / z, float(m + np.log(z))


def beam_attention(q: np.ndarray, ctx_k: np.ndarray, ctx_v: np.ndarray,
                   beam_k: Sequence[np.ndarray], beam_v: Sequence[np.ndarray],
                   ancestry: Sequence[Sequence[int]], beams: Sequence[int] = None
                   ) -> np.ndarray:
    """Attention output of the live beams of one request at one layer.

    q        [n_beams, Hq, D]        query rows, indexed by beam slot
    ctx_k/v  [Hkv, T, D]             the request's context keys / values
    beam_k/v list over levels j < t of [W, Hkv, D]: K/V of the token chosen at
             level j, stored at the slot the beam had after step j
    ancestry ancestry[b][j] = slot at level j on beam b's path (j < t)
    beams    slots to evaluate (default: every row of ``q``)

    Returns float64 [len(beams), Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    n_q_heads, d = q.shape[1], q.shape[2]
    n_kv_heads = ctx_k.shape[0]
    group = n_q_heads // n_kv_heads
    scale = 1.0 / np.sqrt(d)
    if beams is None:
        beams = range(q.shape[0])
    out = np.zeros((len(beams), n_q_heads, d), dtype=np.float64)
    for i, b in enumerate(beams):
        path = ancestry[b]
        for qh in range(n_q_heads):
            kvh = qh // group
            ks = [np.asarray(ctx_k[kvh], dtype=np.float64)]
            vs = [np.asarray(ctx_v[kvh], dtype=np.float64)]
            for j, slot in enumerate(path):
                ks.append(np.asarray(beam_k[j][slot, kvh], dtype=np.float64)[None, :])
                vs.append(np.asarray(beam_v[j][slot, kvh], dtype=np.float64)[None, :])
            keys = np.concatenate(ks, axis=0)
            values = np.concatenate(vs, axis=0)
            out[i, qh], _ = attend_row(q[b, qh], keys, values, scale)
    return out

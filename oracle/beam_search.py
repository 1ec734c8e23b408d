"""Item-constrained wide beam search over semantic-ID codes (oracle, test infrastructure).

What one step computes, read from the pages:
  * [GRINF] section "Background: what inference a recommendation request
    needs": beam search keeps the highest-scoring prefixes, expands and
    prunes them at each step, and every beam that survives the last step is
    returned (not only the best one).
  * [RECSYS] section "语义ID：解决稀疏性与长尾问题": the output logits give the
    ranking.  Section "语义ID生成式推荐专用推理框架": item-constrained top-K,
    dynamic beam width, beam ancestry (BeamPath).

Readings where the pages are silent (each is listed in the design notes):
  1. log-probabilities are the full-vocabulary log-softmax of the logit row;
     invalid codes are then excluded, with no renormalisation over the
     allowed codes;
  2. a beam's score is the sum of its code log-probabilities (every item has
     the same length, so no length penalty); one root beam of score 0;
  3. the level-t code c is vocabulary token ``code_base + t*C + c``;
  4. candidates of a step are all (beam b, code c) with c valid after b's
     prefix; key = S_b + lp_b[token(t, c)]; they are ordered by key
     descending, then by flat index f = b*C + c ascending, and the first
     min(W, #candidates) survive -- this is the new beam width (dynamic
     width); the survivor of rank i takes slot i;
  5. float keys: ``key_mode="f64"`` adds in float64; ``key_mode="f32"``
     evaluates key32 = S32 + (x32 - LSE32) with one float32 rounding per
     operation (the contract under which selections compare bit for bit).
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

from .trie import Trie


def token_id(level: int, code: int, code_base: int, codes_per_level: int) -> int:
    """Vocabulary id of code ``code`` at level ``level`` (reading 3)."""
    return code_base + level * codes_per_level + code


def log_softmax_row(x: np.ndarray) -> Tuple[np.ndarray, float]:
    """Full-vocabulary log-softmax of one logit row in float64.

    Returns (log-probabilities [V], natural-log log-sum-exp).
    """
    x = np.asarray(x, dtype=np.float64)
    m = x.max()
    lse = m + np.log(np.exp(x - m).sum())
    return x - lse, float(lse)


def key_f32(score32, x32, lse32) -> np.float32:
    """key32 = S32 + (x32 - LSE32), each operation rounded once to float32."""
    d = np.float32(np.float32(x32) - np.float32(lse32))
    return np.float32(np.float32(score32) + d)


def ordered_f32(v) -> int:
    """Total-order integer of a float32 value (larger float -> larger int).

    Used by tests to express "identical fp32 keys" as integer equality; -0.0
    maps to the same integer as +0.0.
    """
    v = np.float32(v)
    if v == 0:
        v = np.float32(0.0)
    u = int(np.array([v], dtype=np.float32).view(np.uint32)[0])
    return (u | 0x80000000) if (u & 0x80000000) == 0 else (~u) & 0xFFFFFFFF


def rank_candidates(cands: list) -> list:
    """Order candidates (key, flat, b, c) by key descending, then flat index
    ascending (reading 4); the order is total, so the selection is unique."""
    return sorted(cands, key=lambda e: (-float(e[0]), e[1]))


class OracleBeam:
    """Beam state of one request plus the sort-based constrained step.

    State per level t (after step t): ``parents[t][i]`` (slot at level t-1,
    0 = root for t = 0), ``codes[t][i]``, ``scores[t][i]``.  This is the
    BeamPath: a beam's code string is recovered by following parents.
    """

    def __init__(self, trie: Trie, width: int, n_levels: int, codes_per_level: int,
                 code_base: int, key_mode: str = "f64"):
        if key_mode not in ("f64", "f32"):
            raise ValueError(key_mode)
        self.trie = trie
        self.width = int(width)
        self.n_levels = int(n_levels)
        self.C = int(codes_per_level)
        self.code_base = int(code_base)
        self.key_mode = key_mode
        self.parents: List[List[int]] = []
        self.codes: List[List[int]] = []
        self.scores: List[list] = []

    # -- beam bookkeeping ---------------------------------------------------
    @property
    def t(self) -> int:
        return len(self.codes)

    def n_live(self) -> int:
        return 1 if self.t == 0 else len(self.codes[-1])

    def ancestry(self) -> List[List[int]]:
        """For each live beam b: slot on its path at levels 0..t-1."""
        if self.t == 0:
            return [[]]
        out = []
        for b in range(self.n_live()):
            path = [b]
            for lvl in range(self.t - 1, 0, -1):
                path.append(self.parents[lvl][path[-1]])
            out.append(path[::-1])
        return out

    def prefixes(self) -> List[Tuple[int, ...]]:
        return [tuple(self.codes[j][a] for j, a in enumerate(path)) for path in self.ancestry()]

    def beam_scores(self) -> list:
        if self.t == 0:
            return [np.float32(0.0) if self.key_mode == "f32" else 0.0]
        return list(self.scores[-1])

    # -- one step ---------------------------------------------------------------
    def step(self, logits: np.ndarray, lse_in: Optional[Sequence[float]] = None) -> Dict:
        """Select level-``t`` codes from per-beam logit rows.

        logits  [>= n_live, V] rows by beam slot (float32 or float64 values)
        lse_in  optional per-beam log-sum-exp to use instead of the oracle's
                own (float32 values; only meaningful with key_mode="f32")
        Returns a dict with per-beam ``lse`` (float64 unless overridden),
        ``logprobs`` [n_live, C] float64 -- the level's C code entries of each
        row's full-vocabulary log-softmax, for every code, valid or not (the
        candidate list says which codes are valid) -- the ordered candidate
        list and the selection.
        """
        t = self.t
        if t >= self.n_levels:
            raise RuntimeError("all levels already decoded")
        n = self.n_live()
        prefixes = self.prefixes()
        S = self.beam_scores()
        lo = token_id(t, 0, self.code_base, self.C)
        lse_out = []
        lp_out = np.full((n, self.C), -np.inf, dtype=np.float64)
        cands = []  # (key, flat, b, c)
        for b in range(n):
            row = np.asarray(logits[b])
            lp, lse = log_softmax_row(row)
            lp_out[b] = lp[lo:lo + self.C]
            if lse_in is not None:
                lse_used = np.float32(lse_in[b])
            else:
                lse_used = lse
            lse_out.append(lse_used)
            for c in self.trie.valid_codes(prefixes[b]):
                x = row[lo + c]
                if self.key_mode == "f32":
                    key = key_f32(S[b], np.float32(x), np.float32(lse_used))
                    if key == 0:
                        key = np.float32(0.0)
                else:
                    key = float(S[b]) + (float(x) - float(lse_used))
                cands.append((key, b * self.C + c, b, c))
        cands = rank_candidates(cands)
        keep = cands[: self.width]
        self.parents.append([e[2] for e in keep])
        self.codes.append([e[3] for e in keep])
        self.scores.append([e[0] for e in keep])
        return {"lse": lse_out, "logprobs": lp_out, "candidates": cands, "selected": keep,
                "n_valid": len(cands)}

    # -- results --------------------------------------------------------------
    def results(self) -> List[Tuple[Tuple[int, ...], Optional[int], float]]:
        """Every surviving beam in rank order: (code tuple, item id, score)."""
        out = []
        for pre, s in zip(self.prefixes(), self.beam_scores()):
            out.append((pre, self.trie.item(pre), s))
        return out


def exhaustive_scores(trie: Trie, logits_of_prefix: Callable[[Tuple[int, ...]], np.ndarray],
                      code_base: int, codes_per_level: int) -> Dict[Tuple[int, ...], float]:
    """Score of every item by brute force: sum over levels of the code's
    full-vocabulary log-probability given the item's own prefix (float64)."""
    cache: Dict[Tuple[int, ...], np.ndarray] = {}
    out = {}
    for tup, _ in trie.items():
        total = 0.0
        for t, c in enumerate(tup):
            pre = tup[:t]
            if pre not in cache:
                cache[pre], _ = log_softmax_row(logits_of_prefix(pre))
            total += cache[pre][token_id(t, c, code_base, codes_per_level)]
        out[tup] = total
    return out

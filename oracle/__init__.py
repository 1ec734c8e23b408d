"""CPU oracle for the wide-beam semantic-ID decode step (test infrastructure).

This package is a plain, slow, float64 restatement of what one decode step
computes.  It is test infrastructure: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  It shares no code,
table or helper with the CUDA library in ``beam_decode_gb300`` and imports
nothing from it; the two meet only through the seeded inputs of
``beam_decode_gb300.workload``, which hold none of the method's arithmetic.

Sources (the pages carry no formulas, listings or worked examples; every
step below is the plainest reading of their prose):

[GRINF] "Advancing Generative Recommendation Inference: our collaboration
    with NVIDIA on TensorRT LLM" (English summary page).
    - section "Background: what inference a recommendation request needs":
      an item is a short string of semantic IDs generated one token at a
      time; beam search keeps the highest-scoring prefixes, expands and
      prunes them at each step, and returns every surviving beam, not only
      the best one.
    - section "Scoring many candidates at once": multi-item scoring -- user
      prefix and every candidate in one sequence, a mask that lets each
      candidate see only the prefix and itself, label-token log-probabilities
      read out, candidates ranked by them.
[RECSYS] zhiding.cn article on NVIDIA recsys-examples and nv-embedding-cache.
    - section "语义ID：解决稀疏性与长尾问题" (semantic IDs): decoding semantic
      IDs yields the recommendation directly, and the output logits give the
      ranking.
    - section "语义ID生成式推荐专用推理框架" (semantic-ID GR inference
      framework): long shared request context (ContextKV), short per-beam
      decode history (BeamKV), beam ancestry (BeamPath), dynamic beam width,
      item-constrained generation / item-constrained top-K.

Modules:
    trie         -- dict trie of valid code prefixes (item constraint)
    attention    -- per-beam attention over the concatenated context+beam sequence
    beam_search  -- full-vocabulary log-softmax, constrained candidate
                    enumeration, sort-based selection, beam state and results
    scoring      -- multi-item scoring: masked attention of candidate tokens,
                    label-token log-probabilities, ranking

Parity pins: see tests/test_oracle_*.py.  Every function here is pinned by a
library routine, a closed form, brute-force enumeration, an invariant, or a
hand-worked fixture under tests/golden/.
"""
from .trie import Trie
from .attention import attend_row, beam_attention
from .beam_search import (log_softmax_row, OracleBeam, exhaustive_scores, token_id,
                          key_f32, ordered_f32)
from .scoring import label_logprobs, multi_item_attention, rank, segment_rows

__all__ = ["Trie", "attend_row", "beam_attention", "log_softmax_row", "OracleBeam",
           "exhaustive_scores", "token_id", "key_f32", "ordered_f32", "label_logprobs",
           "multi_item_attention", "rank", "segment_rows"]

"""Seeded synthetic inputs for the wide-beam semantic-ID decode step.

This module draws random numbers and nothing else: item catalogues (code
tuples), query / key / value tensors and logit rows.  It holds none of the
method's arithmetic (no softmax, no attention, no selection, no trie walk),
so both the CUDA path (through the tests and the bench) and the CPU oracle
may be fed from it.

Workload shapes follow the pages:
  * "Advancing Generative Recommendation Inference: our collaboration with
    NVIDIA on TensorRT LLM", section "Performance: how to read the two
    benchmark charts": prompt 2,000 tokens, 5 generated tokens, beam 30,
    Qwen3-1.7B.
  * zhiding.cn article on NVIDIA recsys-examples, section
    "语义ID生成式推荐专用推理框架" (semantic-ID GR inference framework):
    context 1,000 and 5,000 tokens, beam 256, 3 output tokens, Qwen3-1.7B;
    thousands of history tokens, 2-3 decoded semantic-ID tokens, beam 128
    or 256.
Qwen3-1.7B attention geometry: 28 layers, 16 query heads, 8 KV heads,
head_dim 128, vocabulary 151,936.  No weights are used: every tensor is
drawn from a seeded normal distribution.

Streams: host arrays come from ``numpy.random.default_rng([seed, tag])``;
device tensors from ``torch.Generator(device).manual_seed(seed*1000+tag)``.
Each tensor kind has its own ``tag`` so that changing one size does not
shift another tensor's values.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

# stream tags: one per tensor kind
TAG_Q = 1
TAG_CTX_K = 2
TAG_CTX_V = 3
TAG_BEAM_K = 4
TAG_BEAM_V = 5
TAG_LOGITS = 6
TAG_CTXLEN = 7
TAG_WIDTH = 8
TAG_STEPS = 9
TAG_TRIE = 99


@dataclasses.dataclass
class Workload:
    """Geometry of one synthetic decode batch."""
    name: str
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    n_levels: int            # semantic-ID length L (code levels)
    codes_per_level: int     # C
    code_base: int           # token id of (level 0, code 0)
    ctx_lens: List[int]      # per request T_r
    beam_widths: List[int]   # per request W_r (maximum width)
    n_items: List[int]       # per request catalogue size (shared catalogue when all equal and shared_trie)
    trie_dist: str           # "uniform" or "zipf"
    shared_trie: bool        # one catalogue for every request
    logit_std: float = 2.0
    seed: int = 1
    dtype: str = "bf16"      # storage type of Q/K/V on the device

    @property
    def n_requests(self) -> int:
        return len(self.ctx_lens)

    @property
    def rows(self) -> int:
        return int(sum(self.beam_widths))

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


def _qwen3_geometry() -> dict:
    return dict(n_layers=28, n_q_heads=16, n_kv_heads=8, head_dim=128, vocab=151936)


def make_workload(name: str, seed: Optional[int] = None) -> Workload:
    """Return one of the named workloads.

    ``tiny``   1 request, 1 layer, 2 q heads / 1 KV head, head_dim 64, context
               64, beam 4, 2 code levels x 16 codes (token ids 512..543),
               vocab 1024, 50 items drawn uniformly.
    ``page1``  64 requests, context 2000, beam 30, 5 levels x 256 codes,
               200k uniform items.
    ``short``  16 requests, context 1000, beam 256, 3 levels x 256, 1M Zipf(1.1) items.
    ``long``   8 requests, context 5000, beam 256, 3 levels x 256, 1M uniform items.
    ``mixed``  32 requests, context U[500, 5000], beam in {32,64,128,256},
               3..5 levels, per-request catalogues of 100k..1M items.
    """
    if name == "tiny":
        s = 0 if seed is None else seed
        return Workload("tiny", n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=64,
                        vocab=1024, n_levels=2, codes_per_level=16, code_base=512,
                        ctx_lens=[64], beam_widths=[4], n_items=[50], trie_dist="uniform",
                        shared_trie=True, seed=s)
    s = 1 if seed is None else seed
    g = _qwen3_geometry()
    if name == "page1":
        L, C = 5, 256
        return Workload("page1", **g, n_levels=L, codes_per_level=C, code_base=g["vocab"] - L * C,
                        ctx_lens=[2000] * 64, beam_widths=[30] * 64, n_items=[200_000] * 64,
                        trie_dist="uniform", shared_trie=True, seed=s)
    if name == "short":
        L, C = 3, 256
        return Workload("short", **g, n_levels=L, codes_per_level=C, code_base=g["vocab"] - L * C,
                        ctx_lens=[1000] * 16, beam_widths=[256] * 16, n_items=[1_000_000] * 16,
                        trie_dist="zipf", shared_trie=True, seed=s)
    if name == "long":
        L, C = 3, 256
        return Workload("long", **g, n_levels=L, codes_per_level=C, code_base=g["vocab"] - L * C,
                        ctx_lens=[5000] * 8, beam_widths=[256] * 8, n_items=[1_000_000] * 8,
                        trie_dist="uniform", shared_trie=True, seed=s)
    if name == "mixed":
        rng = np.random.default_rng([s, TAG_CTXLEN])
        ctx = [int(v) for v in rng.integers(500, 5001, size=32)]
        rngw = np.random.default_rng([s, TAG_WIDTH])
        widths = [int(v) for v in rngw.choice([32, 64, 128, 256], size=32)]
        rngn = np.random.default_rng([s, TAG_STEPS])
        items = [int(v) for v in rngn.integers(100_000, 1_000_001, size=32)]
        # one level count for the batch: the C-ABI handle has one code layout;
        # 3..5 levels are drawn once per batch
        L = int(rngn.integers(3, 6))
        C = 256
        return Workload("mixed", **g, n_levels=L, codes_per_level=C, code_base=g["vocab"] - L * C,
                        ctx_lens=ctx, beam_widths=widths, n_items=items,
                        trie_dist="zipf", shared_trie=False, seed=s)
    raise KeyError(name)


# ----------------------------------------------------------------------------
# item catalogues (code tuples)
# ----------------------------------------------------------------------------

def _zipf_probs(n: int, a: float) -> np.ndarray:
    ranks = np.arange(1, n + 1, dtype=np.float64)
    w = ranks ** (-a)
    return w / w.sum()


def draw_items(n_items: int, n_levels: int, codes_per_level: int, dist: str = "uniform",
               seed: int = 0, stream: Sequence[int] = ()) -> np.ndarray:
    """Draw ``n_items`` distinct code tuples, int32 ``[n_items, n_levels]``.

    Codes are drawn independently per level, uniformly or Zipf(1.1) over ranks
    1..C with a seeded rank->code permutation per level.  Batches are drawn,
    de-duplicated and appended in order of first appearance until enough
    distinct tuples exist.
    """
    C = codes_per_level
    total = float(C) ** n_levels
    if n_items > total:
        raise ValueError(f"{n_items} distinct items do not fit in {C}^{n_levels} code tuples")
    rng = np.random.default_rng([seed, TAG_TRIE, *stream])
    if dist == "zipf":
        p = _zipf_probs(C, 1.1)
        perms = [rng.permutation(C) for _ in range(n_levels)]
    elif dist != "uniform":
        raise ValueError(dist)
    seen = np.zeros(0, dtype=np.int64)
    order = np.zeros(0, dtype=np.int64)
    batch = max(4 * n_items, 1024)
    draws = 0
    while True:
        cols = []
        for lvl in range(n_levels):
            if dist == "zipf":
                r = rng.choice(C, size=batch, p=p)
                cols.append(perms[lvl][r].astype(np.int64))
            else:
                cols.append(rng.integers(0, C, size=batch, dtype=np.int64))
        key = np.zeros(batch, dtype=np.int64)
        for c in cols:
            key = key * C + c
        allkeys = np.concatenate([order, key])
        _, first = np.unique(allkeys, return_index=True)
        first.sort()
        order = allkeys[first]
        draws += batch
        if order.size >= n_items:
            order = order[:n_items]
            break
        if draws > 200 * n_items + 10_000_000:
            raise RuntimeError("could not draw enough distinct items")
    out = np.empty((n_items, n_levels), dtype=np.int32)
    k = order.copy()
    for lvl in range(n_levels - 1, -1, -1):
        out[:, lvl] = (k % C).astype(np.int32)
        k //= C
    return out


def workload_items(w: Workload) -> List[np.ndarray]:
    """Per-request catalogues (the same array object repeated when shared)."""
    if w.shared_trie:
        items = draw_items(w.n_items[0], w.n_levels, w.codes_per_level, w.trie_dist, w.seed)
        return [items] * w.n_requests
    return [draw_items(n, w.n_levels, w.codes_per_level, w.trie_dist, w.seed, stream=(r,))
            for r, n in enumerate(w.n_items)]


# ----------------------------------------------------------------------------
# dense tensors
# ----------------------------------------------------------------------------

def host_normal(shape, seed: int, tag: int, sub: Sequence[int] = (), std: float = 1.0) -> np.ndarray:
    """float32 normal draws from ``default_rng([seed, tag, *sub])``."""
    rng = np.random.default_rng([seed, tag, *sub])
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bfloat16 (ties to even); returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16
    out = (u.astype(np.uint32) << 16).view(np.float32)
    return out.reshape(x.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are exactly bfloat16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def device_normal(shape, seed: int, tag: int, device, dtype=None, std: float = 1.0, sub: int = 0):
    """Normal draws on ``device`` from ``torch.Generator(device).manual_seed(seed*1000+tag)``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000 + int(tag) + 1_000_003 * int(sub))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if dtype is not None:
        x = x.to(dtype)
    return x

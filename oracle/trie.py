"""Item constraint as a plain dictionary trie (oracle, test infrastructure).

[RECSYS] section "语义ID生成式推荐专用推理框架": generation is constrained to
items ("物品约束生成", item-constrained top-K).  [GRINF] section "Background":
each item is a short string of semantic IDs, and a generated code string is
mapped back to the item.

Reading: an item is a tuple of L codes, one per level, each code in
[0, C).  A prefix of length t admits code c at level t iff some item starts
with prefix + (c,).  Items must be distinct tuples.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np


class Trie:
    """Valid-prefix sets and the item map, held in Python dicts."""

    def __init__(self, codes: np.ndarray, item_ids: Optional[Sequence[int]] = None,
                 codes_per_level: Optional[int] = None):
        codes = np.asarray(codes)
        if codes.ndim != 2:
            raise ValueError("codes must be [n_items, n_levels]")
        self.n_levels = int(codes.shape[1])
        self.codes_per_level = codes_per_level
        if item_ids is None:
            item_ids = range(codes.shape[0])
        self._next: Dict[Tuple[int, ...], set] = {}
        self._item: Dict[Tuple[int, ...], int] = {}
        for row, iid in zip(codes.tolist(), item_ids):
            tup = tuple(int(c) for c in row)
            if codes_per_level is not None and any(c < 0 or c >= codes_per_level for c in tup):
                raise ValueError(f"code out of range in item {tup}")
            if tup in self._item:
                raise ValueError(f"duplicate item {tup}")
            self._item[tup] = int(iid)
            for t in range(self.n_levels):
                self._next.setdefault(tup[:t], set()).add(tup[t])
        self._sorted: Dict[Tuple[int, ...], List[int]] = {k: sorted(v) for k, v in self._next.items()}

    def valid_codes(self, prefix: Sequence[int]) -> List[int]:
        """Codes that extend ``prefix`` towards at least one item (ascending)."""
        return self._sorted.get(tuple(prefix), [])

    def item(self, tup: Sequence[int]) -> Optional[int]:
        return self._item.get(tuple(tup))

    def items(self) -> Iterable[Tuple[Tuple[int, ...], int]]:
        return self._item.items()

    def frontier_sizes(self) -> List[int]:
        """Number of distinct valid prefixes of length t+1, for t = 0..L-1."""
        out = []
        for t in range(self.n_levels):
            out.append(len({tup[: t + 1] for tup in self._item}))
        return out

    def __len__(self) -> int:
        return len(self._item)

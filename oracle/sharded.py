"""Key-sharded top-k -- TEST INFRASTRUCTURE ONLY (numpy / plain Python).

The GLM5 LoRA blog (section 3.1, 训练侧: context parallelism for long sequences) splits
a sequence over devices and reports that a top-k taken on each shard alone agrees with
the full-sequence top-k only 68 % of the time, against 99.97 % once the shards'
indexer results are gathered (THD layout plus an AllGather).  The exact form of that
gather, taken here: every shard of keys keeps its own best ``min(k, visible)`` keys as
(score, global key index) candidates, ordered by (score desc, index asc) and padded
with (-inf, -1); the candidates of all shards are gathered; the best
``min(topk_limit, visible)`` of their union under the same order are the top-k of the
whole row.  Nothing is lost: a key among the row's best k is among the best k of its
own shard, because every key that beats it inside its shard also beats it in the row.

``shard_candidates`` and ``merge_candidates`` are that definition written out with a
full sort per row; ``tests/test_oracle_pins.py`` pins them against the dense oracle's
own full-row top-k, brute-force ranks on tiny rows, and their invariants.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

ORDER_SCORE = 0
ORDER_INDEX = 1


def _sorted_pairs(pairs):
    """(score, index) pairs by score descending, then index ascending (-0.0 == +0.0)."""
    return sorted(pairs, key=lambda p: (-float(p[0]), int(p[1])))


def shard_candidates(scores: np.ndarray, n_visible: Sequence[int], key_offset: int, shard_len: int,
                     k_cand: int):
    """Candidates of the shard holding keys key_offset .. key_offset + shard_len - 1.

    scores [T, >= key_offset + shard_len]: each row's scores at global key positions;
    row t sees keys 0 .. n_visible[t] - 1.  Returns (cand_scores [T, k_cand] fp64 with -inf
    padding, cand_idx [T, k_cand] int32 global indices with -1 padding)."""
    T = scores.shape[0]
    cs = np.full((T, k_cand), -np.inf, dtype=np.float64)
    ci = np.full((T, k_cand), -1, dtype=np.int32)
    for t in range(T):
        hi = min(key_offset + shard_len, int(n_visible[t]))
        pairs = [(scores[t, s], s) for s in range(key_offset, hi)]
        best = _sorted_pairs(pairs)[:k_cand]
        for i, (v, s) in enumerate(best):
            cs[t, i] = v
            ci[t, i] = s
    return cs, ci


def merge_candidates(cand_scores: np.ndarray, cand_idx: np.ndarray, topk_limit: int, k_out: int,
                     order: int = ORDER_SCORE) -> np.ndarray:
    """Top-k of the union of the shards' candidates.

    cand_scores / cand_idx [n_shards, T, k_cand] (entries with index -1 are padding).
    Returns int32 [T, k_out]: min(topk_limit, valid candidates, k_out) indices by
    (score desc, index asc) -- or ascending index for ORDER_INDEX -- then -1."""
    n_shards, T, _ = cand_idx.shape
    out = np.full((T, k_out), -1, dtype=np.int32)
    for t in range(T):
        pairs = [(cand_scores[j, t, i], cand_idx[j, t, i]) for j in range(n_shards)
                 for i in range(cand_idx.shape[2]) if cand_idx[j, t, i] >= 0]
        keep = min(topk_limit, len(pairs), k_out)
        sel = [int(s) for _, s in _sorted_pairs(pairs)[:keep]]
        if order == ORDER_INDEX:
            sel = sorted(sel)
        out[t, :keep] = sel
    return out

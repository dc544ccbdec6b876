"""Oracle: the -1 padded top-k lists the decode consumes (TEST INFRASTRUCTURE).

"Prime Intellect unveils Prime Inference", section "4-bit caches open the
way", item 3: every query token's list has 2048 slots, the empty ones padded
so they contribute nothing. "Prime Inference: Fast, Reliable Serving for
Frontier Open Models", section "A native NVFP4 sparse-MLA decode kernel": the
decode consumes the positions the sparse indexer selected. The indexer's
scores need trained weights the pages do not give; they are an input here.

Readings (the pages give neither): equal scores rank by lower position; the
chosen positions are listed in increasing order, then -1; -0.0 ranks as
+0.0. Only tests, the package smoke check and the bench's CPU baseline may
use this package.
"""
from __future__ import annotations

import numpy as np


def topk_select(scores, topk: int, lengths=None) -> np.ndarray:
    """scores [T, ncols] (real); row t's candidates are positions
    0 .. lengths[t] - 1 (all ncols when lengths is None; clamped to
    [0, ncols]). Returns int64 [T, topk]."""
    s = np.asarray(scores, dtype=np.float64)
    if np.isnan(s).any():
        raise ValueError("NaN scores")
    T, ncols = s.shape
    out = np.full((T, topk), -1, dtype=np.int64)
    for t in range(T):
        L = ncols if lengths is None else int(min(max(int(lengths[t]), 0), ncols))
        k = min(topk, L)
        pos = np.arange(L)
        # rank by score descending, then position ascending (lexsort: last key first);
        # + 0.0 turns -0.0 into +0.0
        order = np.lexsort((pos, -(s[t, :L] + 0.0)))
        out[t, :k] = np.sort(pos[order[:k]])
    return out

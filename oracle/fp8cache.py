"""Oracle: the FP8 cache the NVFP4 format is measured against (TEST
INFRASTRUCTURE).

"Prime Inference: Fast, Reliable Serving for Frontier Open Models", section
"Making room for low-latency decode": an FP8 row is 576 bytes, the 512 latent
and 64 RoPE values one byte each. "Prime Inference open-model serving",
section "KV 캐시와 데이터 전송": the FP8 decode is the comparator of the NVFP4
decode (13.7 against 12.0 us).

Readings (the pages give the size only): latent bytes first, then RoPE; each
value is E4M3(v), nearest even, saturating, no scale; the cache is
[num_pages, 64, 576] with the one-layer slot rule. The decode is
``attention.attend`` over the decoded rows. Only tests, the package smoke
check and the bench's CPU baseline may use this package.
"""
from __future__ import annotations

import numpy as np

from . import formats
from .attention import _as_np, attend, select_rows

FP8_ROW = 576
LATENT = 512


def pack_rows(latent, rope) -> np.ndarray:
    """576-byte rows of N tokens: latent [N, 512], rope [N, 64] (finite reals)."""
    latent = np.asarray(latent, dtype=np.float64)
    rope = np.asarray(rope, dtype=np.float64)
    row = np.empty((latent.shape[0], FP8_ROW), dtype=np.uint8)
    row[:, :LATENT] = formats.e4m3_encode(latent)
    row[:, LATENT:] = formats.e4m3_encode(rope)
    return row


def pack_into_cache(latent, rope, slot_mapping, cache: np.ndarray) -> np.ndarray:
    """Write N tokens' rows into cache [num_pages, 64, 576] (in place,
    returned); negative slots are skipped."""
    slot_mapping = np.asarray(slot_mapping, dtype=np.int64)
    flat = cache.reshape(-1, FP8_ROW)
    keep = slot_mapping >= 0
    if np.any(slot_mapping[keep] >= flat.shape[0]):
        raise IndexError("slot beyond the cache")
    flat[slot_mapping[keep]] = pack_rows(np.asarray(latent)[keep], np.asarray(rope)[keep])
    return cache


def unpack_rows(rows: np.ndarray):
    """[N, 576] -> (latent float64 [N, 512], rope float64 [N, 64])."""
    rows = np.asarray(rows, dtype=np.uint8)
    return formats.e4m3_decode(rows[:, :LATENT]), formats.e4m3_decode(rows[:, LATENT:])


def sparse_mla_decode(q_latent, q_rope, cache, block_table, topk_idx, sm_scale, q_seq_idx=None, seq_lens=None,
                      tokens=None):
    """The oracle decode over an FP8 cache -> (out [T', H, 512], lse [T', H], n_bad)."""
    ql = _as_np(q_latent, np.float64)
    qr = _as_np(q_rope, np.float64)
    cache = _as_np(cache, np.uint8).reshape(-1, FP8_ROW)
    bt = _as_np(block_table, np.int64)
    topk = _as_np(topk_idx, np.int64)
    qs = _as_np(q_seq_idx, np.int64)
    sl = _as_np(seq_lens, np.int64)
    T = ql.shape[0]
    toks = range(T) if tokens is None else list(tokens)
    outs, lses, n_bad = [], [], 0
    for t in toks:
        b = 0 if qs is None else int(qs[t])
        L = None if sl is None or not 0 <= b < bt.shape[0] else int(sl[b])
        slots, bad = select_rows(topk[t], b, bt, L, cache.shape[0])
        n_bad += bad
        K_lat, K_rope = unpack_rows(cache[slots])
        o, l = attend(ql[t], qr[t], K_lat, K_rope, sm_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses), n_bad

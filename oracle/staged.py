"""Oracle: the staged baseline (TEST INFRASTRUCTURE).

"Prime Inference open-model serving", section "KV 캐시와 데이터 전송", and
"Prime Intellect unveils Prime Inference", section "4-bit caches open the
way": before the native kernel, the compressed rows were first unpacked into
a temporary FP8 buffer in GPU memory and an existing FP8 attention kernel ran
on that buffer; the extra conversion and memory round trip is what the native
kernel removes. An FP8 row is 576 bytes: 512 latent values + 64 RoPE values,
all E4M3 ("Prime Inference: Fast, Reliable Serving for Frontier Open Models",
section "Making room for low-latency decode").

Stage 1 (reading of an unstated step): every selected NVFP4 row becomes one
576-byte E4M3 row. Latent value d is E2M1(code_d) * scale_{d//16} re-rounded
to E4M3 (nearest even, saturating at 448; up to 6 significant bits and values
up to 2688 do not all fit, so this step is lossy); the RoPE bytes are copied.
Rows go to buf[t, k] in list order; idx[t, k] = k for a valid slot, -1
otherwise, and invalid rows are left as they were.

Stage 2: the attention of ``attention.attend`` over the FP8 rows.
"""
from __future__ import annotations

import numpy as np

from . import formats
from . import pack as _pack
from .attention import _as_np, attend, select_rows

FP8_ROW = 576


def stage_dequant_fp8(cache, block_table, topk_idx, q_seq_idx=None, seq_lens=None):
    """-> (buf uint8 [T, K, 576] with invalid rows zero, idx int32 [T, K])."""
    cache = _as_np(cache, np.uint8).reshape(-1, _pack.ROW_BYTES)
    bt = _as_np(block_table, np.int64)
    topk = _as_np(topk_idx, np.int64)
    qs = _as_np(q_seq_idx, np.int64)
    sl = _as_np(seq_lens, np.int64)
    T, K = topk.shape
    buf = np.zeros((T, K, FP8_ROW), dtype=np.uint8)
    idx = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        b = 0 if qs is None else int(qs[t])
        L = None if sl is None else int(sl[b])
        for k in range(K):
            slots, bad = select_rows(topk[t, k:k + 1], b, bt, L, cache.shape[0])
            if slots.size == 0:
                continue
            lat, _ = _pack.unpack_row(cache[slots[0]])
            buf[t, k, :512] = formats.e4m3_encode(lat)
            buf[t, k, 512:] = cache[slots[0], _pack.ROPE_OFF:_pack.ROW_BYTES]
            idx[t, k] = k
    return buf, idx


def stage_dequant_fp8_fast(cache, block_table, topk_idx, q_seq_idx=None, seq_lens=None):
    """Same result as stage_dequant_fp8, vectorised per token."""
    cache = _as_np(cache, np.uint8).reshape(-1, _pack.ROW_BYTES)
    bt = _as_np(block_table, np.int64)
    topk = _as_np(topk_idx, np.int64)
    qs = _as_np(q_seq_idx, np.int64)
    sl = _as_np(seq_lens, np.int64)
    T, K = topk.shape
    buf = np.zeros((T, K, FP8_ROW), dtype=np.uint8)
    idx = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        b = 0 if qs is None else int(qs[t])
        L = None if sl is None else int(sl[b])
        p = topk[t]
        max_pos = bt.shape[1] * _pack.PAGE_TOKENS
        limit = max_pos if L is None else min(L, max_pos)
        ks = np.nonzero((p >= 0) & (p < limit))[0]
        pv = p[ks]
        slots = bt[b, pv // _pack.PAGE_TOKENS] * _pack.PAGE_TOKENS + pv % _pack.PAGE_TOKENS
        ok = (slots >= 0) & (slots < cache.shape[0])
        ks, slots = ks[ok], slots[ok]
        lat, _ = _pack.unpack_rows(cache[slots])
        buf[t, ks, :512] = formats.e4m3_encode(lat)
        buf[t, ks, 512:] = cache[slots, _pack.ROPE_OFF:_pack.ROW_BYTES]
        idx[t, ks] = ks
    return buf, idx


def decode_fp8rows(q_latent, q_rope, buf, idx, sm_scale, tokens=None):
    """Attention over FP8 rows: key k of token t is buf[t, idx[t, k]] for
    idx[t, k] >= 0. -> (out float64 [T', H, 512], lse float64 [T', H])."""
    ql = _as_np(q_latent, np.float64)
    qr = _as_np(q_rope, np.float64)
    buf = _as_np(buf, np.uint8)
    idx = _as_np(idx, np.int64)
    T = ql.shape[0]
    toks = range(T) if tokens is None else list(tokens)
    outs, lses = [], []
    for t in toks:
        ks = idx[t][idx[t] >= 0]
        rows = buf[t, ks]
        K_lat = formats.e4m3_decode(rows[:, :512])
        K_rope = formats.e4m3_decode(rows[:, 512:])
        o, l = attend(ql[t], qr[t], K_lat, K_rope, sm_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)

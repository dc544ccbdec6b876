"""Oracle: sparse MLA decode attention over an NVFP4 paged cache
(TEST INFRASTRUCTURE).

What is computed ("Prime Inference: Fast, Reliable Serving for Frontier Open
Models", section "A native NVFP4 sparse-MLA decode kernel"; "Prime Intellect
unveils Prime Inference", section "4-bit caches open the way", item 3): each
query token attends only to the positions the sparse indexer selected for it,
reading those compressed rows and unpacking them; the list has 2048 slots and
empty slots are padded so that they contribute nothing. The pages fix FP16
operands with FP32 accumulation for the GPU; the oracle computes the same
definition exactly in float64.

Definition, per query token t and head h (readings listed in the design
notes):

* b = q_seq_idx[t] (0 if absent). A token whose b lies outside the block
  table's rows has no valid slot: every entry other than -1 is a bad index.
* the valid set J(t) holds every slot k whose
  position p = topk_idx[t, k] satisfies 0 <= p < seq_lens[b] (and p inside the
  block table). A slot equal to -1 is padding. Any other out-of-range value
  is also skipped and counted as a bad index. Duplicated positions count
  once per slot.
* the row of position p is slot block_table[b, p // 64] * 64 + p % 64 of the
  cache; K_k = [latent (512) | rope (64)], V_k = latent.
* s_k = sm_scale * (q_latent[t, h] . latent_k + q_rope[t, h] . rope_k)
* m = max_k s_k, lse = m + ln(sum_k exp(s_k - m)) (natural log),
  out = sum_k exp(s_k - lse) V_k.
* J(t) empty: out = 0, lse = -inf.

Outputs are float64; the CUDA path rounds out to bf16 and keeps lse in fp32.
"""
from __future__ import annotations

import numpy as np

from . import pack as _pack

PAGE_TOKENS = 64


def _as_np(x, dtype=None):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (bf16 has no numpy dtype)
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=dtype)


def select_rows(topk_row, seq, block_table, seq_len, num_slots):
    """Physical slots of the valid entries of one token's list.

    Returns (slots [n] int64, n_bad) where n_bad counts entries that are
    neither -1 nor a valid position."""
    p = np.asarray(topk_row, dtype=np.int64)
    if not 0 <= seq < block_table.shape[0]:
        return np.zeros(0, dtype=np.int64), int((p != -1).sum())
    max_pos = block_table.shape[1] * PAGE_TOKENS
    limit = max_pos if seq_len is None else min(int(seq_len), max_pos)
    valid = (p >= 0) & (p < limit)
    bad = (~valid) & (p != -1)
    pv = p[valid]
    slots = block_table[seq, pv // PAGE_TOKENS].astype(np.int64) * PAGE_TOKENS + pv % PAGE_TOKENS
    bad_slot = (slots < 0) | (slots >= num_slots)
    if np.any(bad_slot):
        slots = slots[~bad_slot]
    return slots, int(bad.sum() + bad_slot.sum())


def attend(q_lat, q_rope, K_lat, K_rope, sm_scale):
    """Softmax attention of H query heads over n keys, float64.

    q_lat [H, 512], q_rope [H, 64], K_lat [n, 512], K_rope [n, 64]
    -> out [H, 512], lse [H]."""
    H = q_lat.shape[0]
    if K_lat.shape[0] == 0:
        return np.zeros((H, K_lat.shape[1]), dtype=np.float64), np.full(H, -np.inf)
    s = sm_scale * (q_lat @ K_lat.T + q_rope @ K_rope.T)  # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    L = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(L))[:, 0]
    out = (e / L) @ K_lat
    return out, lse


def sparse_mla_decode(q_latent, q_rope, cache, block_table, topk_idx, sm_scale,
                      q_seq_idx=None, seq_lens=None, tokens=None):
    """Oracle decode. Returns (out float64 [T', H, 512], lse float64 [T', H],
    n_bad) for the tokens listed in `tokens` (default: all, in order).

    cache: uint8 [num_pages, 64, 352]."""
    ql = _as_np(q_latent, np.float64)
    qr = _as_np(q_rope, np.float64)
    cache = _as_np(cache, np.uint8).reshape(-1, _pack.ROW_BYTES)
    bt = _as_np(block_table, np.int64)
    topk = _as_np(topk_idx, np.int64)
    qs = _as_np(q_seq_idx, np.int64)
    sl = _as_np(seq_lens, np.int64)
    T, H, _ = ql.shape
    toks = range(T) if tokens is None else list(tokens)
    outs, lses, n_bad = [], [], 0
    for t in toks:
        b = 0 if qs is None else int(qs[t])
        L = None if sl is None or not 0 <= b < bt.shape[0] else int(sl[b])
        slots, bad = select_rows(topk[t], b, bt, L, cache.shape[0])
        n_bad += bad
        K_lat, K_rope = _pack.unpack_rows(cache[slots])
        o, l = attend(ql[t], qr[t], K_lat, K_rope, sm_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses), n_bad

"""Seeded synthetic inputs for the NVFP4 sparse-MLA pack and decode calls.

This module only draws random numbers and lays them out as the calls'
arguments. It holds none of the method's arithmetic: no quantisation, no
attention, no reading of the cache. Tests, the benchmark and the oracle all
take their inputs from here, so the CUDA path and the oracle see the same
bytes.

Shapes and value distributions follow the workloads the source pages describe
("Prime Inference: Fast, Reliable Serving for Frontier Open Models",
sections "Workload" and "Making room for low-latency decode"; the wireai.ir
article on Prime Inference, section "4-bit caches open the way", item 3):

* latent: 512 values per token, N(0, 1) times a per-channel scale drawn once
  per workload from LogNormal(0, 0.5); RoPE part: 64 values per token, N(0, 1);
  queries: N(0, 1). All are rounded to bf16.
* cache pages hold 64 tokens; logical pages map to physical pages through a
  shuffled block table.
* each query token carries a 2048-slot list of selected positions; empty
  slots hold -1.

Only cache rows that some query token selects (plus, for the write+read
workload, the freshly packed tail) are ever written: the decode call never
reads any other row, so the rest of the cache stays zero.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

PAGE_TOKENS = 64
LATENT_DIM = 512
ROPE_DIM = 64
ROW_BYTES = 352
TOPK = 2048


@dataclasses.dataclass
class Workload:
    """One synthetic problem. All tensors live on the host (CPU)."""

    name: str
    # query side
    q_latent: torch.Tensor  # [T, H, 512] bf16
    q_rope: torch.Tensor  # [T, H, 64] bf16
    topk_idx: torch.Tensor  # [T, topk] int32 logical positions, -1 = empty slot
    q_seq_idx: torch.Tensor  # [T] int32 sequence of each query token
    sm_scale: float
    # cache side
    seq_lens: torch.Tensor  # [B] int32
    block_table: torch.Tensor  # [B, max_pages] int32 physical page ids
    num_pages: int
    # rows written into the cache before the decode (setup, untimed)
    hist_latent: torch.Tensor  # [Nh, 512] bf16
    hist_rope: torch.Tensor  # [Nh, 64] bf16
    hist_slots: torch.Tensor  # [Nh] int32 physical slots
    # rows written by a timed pack call (write+read workload), else empty
    new_latent: torch.Tensor  # [Nn, 512] bf16
    new_rope: torch.Tensor  # [Nn, 64] bf16
    new_slots: torch.Tensor  # [Nn] int32

    @property
    def T(self) -> int:
        return int(self.q_latent.shape[0])

    @property
    def H(self) -> int:
        return int(self.q_latent.shape[1])

    @property
    def topk(self) -> int:
        return int(self.topk_idx.shape[1])

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    def all_written(self):
        """(latent, rope, slots) of every row written before the decode."""
        lat = torch.cat([self.hist_latent, self.new_latent])
        rope = torch.cat([self.hist_rope, self.new_rope])
        slots = torch.cat([self.hist_slots, self.new_slots])
        return lat, rope, slots


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _block_tables(rng, seq_lens):
    """Shuffled physical pages for every sequence; padding entries are 0."""
    pages = [int(math.ceil(int(n) / PAGE_TOKENS)) for n in seq_lens]
    total = sum(pages)
    perm = rng.permutation(total).astype(np.int32)
    max_pages = max(pages)
    table = np.zeros((len(pages), max_pages), dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, total


def _slots_of(table, seq, pos):
    """Physical slot of logical position `pos` of sequence `seq` (input layout)."""
    return table[seq, pos // PAGE_TOKENS] * PAGE_TOKENS + pos % PAGE_TOKENS


def _distinct(rng, lo, hi, n):
    """n distinct integers drawn uniformly from [lo, hi)."""
    span = hi - lo
    if n > span:
        raise ValueError("not enough positions")
    if span <= 4 * n:
        return (rng.permutation(span)[:n] + lo).astype(np.int64)
    out = np.unique(rng.integers(lo, hi, size=int(n * 1.2) + 16))
    while out.size < n:
        out = np.unique(np.concatenate([out, rng.integers(lo, hi, size=n)]))
    return rng.permutation(out)[:n].astype(np.int64)


def _latent_rows(rng, n, chan_scale, outlier_frac=0.0, outlier_mult=20.0):
    lat = rng.standard_normal((n, LATENT_DIM), dtype=np.float32) * chan_scale[None, :]
    if outlier_frac > 0:
        mask = rng.random((n, LATENT_DIM)) < outlier_frac
        lat = np.where(mask, lat * outlier_mult, lat)
    rope = rng.standard_normal((n, ROPE_DIM), dtype=np.float32)
    if outlier_frac > 0:
        mask = rng.random((n, ROPE_DIM)) < outlier_frac
        rope = np.where(mask, rope * outlier_mult, rope)
    return lat, rope


def _assemble(name, rng, seq_lens, q_seq, topk, H, sm_scale, chan_scale,
              new_positions=None, new_seq=0, new_outliers=0.0):
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    table, total_pages = _block_tables(rng, seq_lens)
    T = len(q_seq)
    # rows the decode will read: every valid selected (seq, pos) pair
    sel = topk >= 0
    seqs = np.broadcast_to(np.asarray(q_seq)[:, None], topk.shape)[sel]
    poss = topk[sel]
    slots = _slots_of(table, seqs, poss)
    hist_slots = np.unique(slots)
    new_slots = np.zeros(0, dtype=np.int64)
    if new_positions is not None:
        new_slots = _slots_of(table, np.full(len(new_positions), new_seq), np.asarray(new_positions))
        hist_slots = np.setdiff1d(hist_slots, new_slots)
    hl, hr = _latent_rows(rng, len(hist_slots), chan_scale)
    nl, nr = _latent_rows(rng, len(new_slots), chan_scale, outlier_frac=new_outliers)
    ql = rng.standard_normal((T, H, LATENT_DIM), dtype=np.float32)
    qr = rng.standard_normal((T, H, ROPE_DIM), dtype=np.float32)
    return Workload(
        name=name,
        q_latent=_bf16(ql), q_rope=_bf16(qr),
        topk_idx=torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)),
        q_seq_idx=torch.from_numpy(np.asarray(q_seq, dtype=np.int32)),
        sm_scale=float(sm_scale),
        seq_lens=torch.from_numpy(seq_lens.astype(np.int32)),
        block_table=torch.from_numpy(table),
        num_pages=int(total_pages),
        hist_latent=_bf16(hl), hist_rope=_bf16(hr),
        hist_slots=torch.from_numpy(hist_slots.astype(np.int32)),
        new_latent=_bf16(nl), new_rope=_bf16(nr),
        new_slots=torch.from_numpy(new_slots.astype(np.int32)),
    )


DEFAULT_SM_SCALE = 1.0 / math.sqrt(192.0)


def tiny(seed: int = 0) -> Workload:
    """1 sequence, 1 query token, 16 heads, 4096-token context, top-256."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chan = rng.lognormal(0.0, 0.5, LATENT_DIM).astype(np.float32)
    ctx, k = 4096, 256
    topk = _distinct(rng, 0, ctx, k)[None, :]
    w = _assemble("tiny", rng, [ctx], [0], topk, 16, DEFAULT_SM_SCALE, chan)
    return w


def decode_point(seed: int = 1, T: int = 15, H: int = 64, ctx: int = 200_000,
                 topk: int = TOPK) -> Workload:
    """The pages' decode point: 15 query tokens of one sequence, 64 heads,
    200K-token context, per-token top-2048 distinct uniform positions."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chan = rng.lognormal(0.0, 0.5, LATENT_DIM).astype(np.float32)
    idx = np.stack([_distinct(rng, 0, ctx, topk) for _ in range(T)])
    return _assemble("decode_point", rng, [ctx], [0] * T, idx, H, DEFAULT_SM_SCALE, chan)


def padded(seed: int = 2, T: int = 35, H: int = 64, ctx: int = 32_768,
           topk: int = TOPK, max_pad_frac: float = 0.6) -> Workload:
    """Padded index lists: each token's 2048 slots have a fraction
    f ~ U[0, 0.6] of randomly placed -1 entries; the rest are distinct
    uniform positions."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chan = rng.lognormal(0.0, 0.5, LATENT_DIM).astype(np.float32)
    idx = np.full((T, topk), -1, dtype=np.int64)
    for t in range(T):
        f = rng.uniform(0.0, max_pad_frac)
        n_valid = topk - int(round(f * topk))
        where = rng.permutation(topk)[:n_valid]
        idx[t, where] = _distinct(rng, 0, ctx, n_valid)
    return _assemble("padded", rng, [ctx], [0] * T, idx, H, DEFAULT_SM_SCALE, chan)


def _clustered(rng, ctx, topk, recent=6144):
    """Half the slots distinct within the last `recent` positions, half
    distinct uniform over the older history."""
    n_recent = min(topk // 2, recent)
    lo = max(0, ctx - recent)
    a = _distinct(rng, lo, ctx, n_recent)
    b = _distinct(rng, 0, lo, topk - n_recent)
    return rng.permutation(np.concatenate([a, b]))


def batched(seed: int = 3, num_seqs: int = 64, H: int = 64, topk: int = TOPK,
            ctx_lo: int = 32_768, ctx_hi: int = 140_000) -> Workload:
    """Batched decode: num_seqs sequences x 1-4 query tokens, context
    U[32K, 140K], clustered top-2048 lists."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chan = rng.lognormal(0.0, 0.5, LATENT_DIM).astype(np.float32)
    lens = rng.integers(ctx_lo, ctx_hi + 1, size=num_seqs)
    per = rng.integers(1, 5, size=num_seqs)
    q_seq = np.repeat(np.arange(num_seqs), per)
    idx = np.stack([_clustered(rng, int(lens[s]), topk) for s in q_seq])
    return _assemble("batched", rng, lens, q_seq, idx, H, DEFAULT_SM_SCALE, chan)


def write_read(seed: int = 4, n_new: int = 6144, ctx: int = 140_000, T: int = 128,
               H: int = 64, topk: int = TOPK) -> Workload:
    """Write+read mix: a 6K-token prefill chunk (1% outliers x20) is packed
    into the fresh tail of a 140K-token cache, then 128 query tokens attend
    with clustered top-2048 lists (half inside the fresh tail)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chan = rng.lognormal(0.0, 0.5, LATENT_DIM).astype(np.float32)
    idx = np.stack([_clustered(rng, ctx, topk, recent=n_new) for _ in range(T)])
    new_pos = np.arange(ctx - n_new, ctx)
    return _assemble("write_read", rng, [ctx], [0] * T, idx, H, DEFAULT_SM_SCALE, chan,
                     new_positions=new_pos, new_seq=0, new_outliers=0.01)


def pack_chunk(seed: int, n: int, num_pages: int, outlier_frac: float = 0.01):
    """A stand-alone pack input: n tokens to distinct random slots of a cache
    of num_pages pages. Returns (latent bf16 [n,512], rope bf16 [n,64],
    slots int32 [n])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chan = np.ones(LATENT_DIM, dtype=np.float32)
    lat, rope = _latent_rows(rng, n, chan, outlier_frac=outlier_frac)
    slots = _distinct(rng, 0, num_pages * PAGE_TOKENS, n)
    return _bf16(lat), _bf16(rope), torch.from_numpy(slots.astype(np.int32))


WORKLOADS = {
    "tiny": tiny,
    "decode_point": decode_point,
    "padded": padded,
    "batched": batched,
    "write_read": write_read,
}


def make(name: str, **kw) -> Workload:
    return WORKLOADS[name](**kw)


def describe(w: Workload) -> dict:
    valid = int((w.topk_idx >= 0).sum())
    return {"workload": w.name, "T": w.T, "H": w.H, "topk": w.topk,
            "num_seqs": w.num_seqs, "max_ctx": int(w.seq_lens.max()),
            "page_tokens": PAGE_TOKENS, "valid_slots": valid,
            "sm_scale": w.sm_scale}

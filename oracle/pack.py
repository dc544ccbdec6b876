"""Oracle: the NVFP4 cache row writer (TEST INFRASTRUCTURE).

What one cache row holds ("Prime Inference: Fast, Reliable Serving for
Frontier Open Models", section "Making room for low-latency decode"; the same
numbers in "Prime Inference open-model serving", section "KV 캐시와 데이터
전송", and in "Prime Intellect unveils Prime Inference", section "4-bit caches
open the way"):

* the 512-value latent as 4-bit values with one FP8 scale per 16 values:
  256 bytes of codes + 32 scale bytes;
* the 64-value positional (RoPE) part as FP8: 64 bytes;
* 352 bytes in all, down from 576 for an all-FP8 row (512 + 64).

Readings where the pages are silent (each listed in the design notes):

* group scale = E4M3(amax / 6), amax the largest magnitude of the 16 values
  and 6 the largest E2M1 magnitude, the real quotient rounded to nearest
  even and saturated;
* codes quantise value / S with S the *stored* (rounded) scale;
* byte j of the code region holds value 2j in bits 0-3 and value 2j+1 in
  bits 4-7; group g's scale is byte 256 + g; RoPE value j is byte 288 + j;
* the RoPE part is a plain saturating E4M3 cast, with no scale (the 352-byte
  budget leaves no room for one), and there is no second-level tensor scale.

Inputs must be finite; the cache is [num_pages, 64, 352] bytes and a token
with a negative slot is skipped.
"""
from __future__ import annotations

import numpy as np

from . import formats

LATENT = 512
ROPE = 64
GROUP = 16
CODE_BYTES = LATENT // 2  # 256
SCALE_OFF = CODE_BYTES  # 256
ROPE_OFF = SCALE_OFF + LATENT // GROUP  # 288
ROW_BYTES = ROPE_OFF + ROPE  # 352
PAGE_TOKENS = 64


def group_scales(latent: np.ndarray) -> np.ndarray:
    """E4M3 scale code of every 16-value group: E4M3(amax / 6).

    latent: float64 [N, 512] -> uint8 [N, 32]."""
    g = np.abs(latent).reshape(latent.shape[0], LATENT // GROUP, GROUP)
    amax = g.max(axis=-1)
    return formats.e4m3_encode_quotient(amax, formats.E2M1_MAX)


def pack_rows(latent, rope) -> np.ndarray:
    """352-byte rows of N tokens. latent [N, 512], rope [N, 64] (any real
    dtype; converted to float64 exactly for bf16 inputs) -> uint8 [N, 352]."""
    latent = np.asarray(latent, dtype=np.float64)
    rope = np.asarray(rope, dtype=np.float64)
    n = latent.shape[0]
    assert latent.shape == (n, LATENT) and rope.shape == (n, ROPE)
    sc = group_scales(latent)  # [N, 32]
    S = formats.e4m3_decode(sc)  # [N, 32]
    S_per_value = np.repeat(S, GROUP, axis=1)  # [N, 512]
    codes = formats.e2m1_encode_scaled(latent, S_per_value)  # [N, 512] 0..15
    row = np.zeros((n, ROW_BYTES), dtype=np.uint8)
    row[:, :CODE_BYTES] = codes[:, 0::2] | (codes[:, 1::2] << 4)
    row[:, SCALE_OFF:ROPE_OFF] = sc
    row[:, ROPE_OFF:ROW_BYTES] = formats.e4m3_encode(rope)
    return row


def pack_into_cache(latent, rope, slot_mapping, cache: np.ndarray) -> np.ndarray:
    """Write the rows of N tokens into a paged cache (in place, returned).

    cache: uint8 [num_pages, 64, 352]; slot s is page s // 64, offset s % 64.
    Negative slots are skipped."""
    slot_mapping = np.asarray(slot_mapping, dtype=np.int64)
    flat = cache.reshape(-1, ROW_BYTES)
    keep = slot_mapping >= 0
    if np.any(slot_mapping[keep] >= flat.shape[0]):
        raise IndexError("slot beyond the cache")
    rows = pack_rows(np.asarray(latent)[keep], np.asarray(rope)[keep])
    flat[slot_mapping[keep]] = rows
    return cache


def unpack_row(row: np.ndarray):
    """Decode one 352-byte row: (latent float64 [512], rope float64 [64]).

    The latent value d is E2M1(code_d) * E4M3(scale_{d // 16})."""
    row = np.asarray(row, dtype=np.uint8)
    codes = np.empty(LATENT, dtype=np.uint8)
    codes[0::2] = row[:CODE_BYTES] & 15
    codes[1::2] = row[:CODE_BYTES] >> 4
    S = formats.e4m3_decode(row[SCALE_OFF:ROPE_OFF])
    latent = formats.e2m1_decode(codes) * np.repeat(S, GROUP)
    rope = formats.e4m3_decode(row[ROPE_OFF:ROW_BYTES])
    return latent, rope


def unpack_rows(rows: np.ndarray):
    """Vectorised unpack_row over [N, 352] -> ([N, 512], [N, 64])."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    codes = np.empty((n, LATENT), dtype=np.uint8)
    codes[:, 0::2] = rows[:, :CODE_BYTES] & 15
    codes[:, 1::2] = rows[:, :CODE_BYTES] >> 4
    S = formats.e4m3_decode(rows[:, SCALE_OFF:ROPE_OFF])
    latent = formats.e2m1_decode(codes) * np.repeat(S, GROUP, axis=1)
    rope = formats.e4m3_decode(rows[:, ROPE_OFF:ROW_BYTES])
    return latent, rope

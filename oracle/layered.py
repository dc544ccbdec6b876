"""Oracle: one layer of a block-major multi-layer cache (TEST INFRASTRUCTURE).

"Prime Inference: Fast, Reliable Serving for Frontier Open Models", section
"Changing the layout to reduce fragmentation": a block-major layout keeps one
block's data for several layers together in memory, so that moving KV takes
fewer, larger copies. "Prime Inference open-model serving", section "KV 캐시와
데이터 전송": its blocks are 64 tokens.

Reading (the pages give the layout's name, block-layer-head-token-channel,
not its bytes): for MLA's single latent head the cache is
uint8 [num_blocks, num_layers, 64, 352], i.e. row (block b, layer l, token i)
starts at byte ((b * num_layers + l) * 64 + i) * 352. Slots keep their
one-layer meaning, slot = b * 64 + i, so one block table serves every layer.

Layer l of such a cache is therefore the array cache[:, l], shaped exactly
like a one-layer cache [num_blocks, 64, 352]; the functions below apply the
one-layer oracle to it. Only tests, the package smoke check and the bench's
CPU baseline may use this package.
"""
from __future__ import annotations

import numpy as np

from . import attention as _att
from . import pack as _pack


def row_byte_offset(block: int, layer: int, token: int, num_layers: int) -> int:
    """Byte offset of row (block, layer, token) from the start of the cache."""
    return ((block * num_layers + layer) * 64 + token) * _pack.ROW_BYTES


def layer_view(cache: np.ndarray, layer: int) -> np.ndarray:
    """Layer `layer` of a [num_blocks, num_layers, 64, 352] cache as a
    (contiguous copy of a) one-layer cache [num_blocks, 64, 352]."""
    if cache.ndim != 4 or cache.shape[2:] != (64, _pack.ROW_BYTES):
        raise ValueError("cache must be [num_blocks, num_layers, 64, 352]")
    if not 0 <= layer < cache.shape[1]:
        raise IndexError("layer outside the cache")
    return np.ascontiguousarray(cache[:, layer])


def pack_into_layered_cache(latent, rope, slot_mapping, cache: np.ndarray, layer: int) -> np.ndarray:
    """Write N tokens' rows into layer `layer` (in place, returned); the
    other layers are left as they are."""
    one = layer_view(cache, layer)
    _pack.pack_into_cache(latent, rope, slot_mapping, one)
    cache[:, layer] = one
    return cache


def sparse_mla_decode_layered(q_latent, q_rope, cache: np.ndarray, layer: int, block_table, topk_idx, sm_scale,
                              q_seq_idx=None, seq_lens=None, tokens=None):
    """The oracle decode over layer `layer`."""
    return _att.sparse_mla_decode(q_latent, q_rope, layer_view(cache, layer), block_table, topk_idx, sm_scale,
                                  q_seq_idx, seq_lens, tokens=tokens)

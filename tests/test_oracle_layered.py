"""Pins for the oracle's block-major multi-layer cache (CPU only).

The layout is pinned to its byte formula by markers (every row of a cache
carries its own (block, layer, token) in its first bytes); packing one layer
is pinned to the one-layer writer (the one-layer cache is the special case
num_layers = 1) and to leaving every other layer's bytes alone; the layered
decode is pinned to the one-layer decode of the same rows.
"""
import numpy as np
import pytest

from oracle import layered, pack
from oracle import attention as oatt


def marker_cache(num_blocks, num_layers):
    c = np.zeros((num_blocks, num_layers, 64, pack.ROW_BYTES), dtype=np.uint8)
    for b in range(num_blocks):
        for l in range(num_layers):
            for i in range(64):
                c[b, l, i, :3] = (b, l, i)
    return c


def test_rows_sit_at_the_layout_formula():
    nb, nl = 3, 5
    c = marker_cache(nb, nl)
    flat = c.reshape(-1)
    for b in range(nb):
        for l in range(nl):
            for i in (0, 17, 63):
                off = layered.row_byte_offset(b, l, i, nl)
                assert off == ((b * nl + l) * 64 + i) * 352
                assert tuple(flat[off:off + 3]) == (b, l, i)
    for l in range(nl):
        v = layered.layer_view(c, l)
        assert v.shape == (nb, 64, 352)
        assert (v[:, :, 1] == l).all()
        assert (v[:, :, 0] == np.arange(nb)[:, None]).all()
        assert (v[:, :, 2] == np.arange(64)[None, :]).all()


def test_layer_outside_the_cache_is_refused():
    c = marker_cache(1, 2)
    with pytest.raises(IndexError):
        layered.layer_view(c, 2)
    with pytest.raises(ValueError):
        layered.layer_view(c[:, 0], 0)


def _tokens(rng, n):
    lat = rng.standard_normal((n, 512)) * rng.lognormal(0.0, 0.5, 512)
    rope = rng.standard_normal((n, 64))
    return lat, rope


def test_one_layer_is_the_one_layer_cache():
    rng = np.random.default_rng(3)
    lat, rope = _tokens(rng, 40)
    slots = rng.choice(4 * 64, 40, replace=False)
    one = np.zeros((4, 64, 352), dtype=np.uint8)
    pack.pack_into_cache(lat, rope, slots, one)
    lay = np.zeros((4, 1, 64, 352), dtype=np.uint8)
    layered.pack_into_layered_cache(lat, rope, slots, lay, 0)
    assert np.array_equal(lay[:, 0], one)


def test_packing_a_layer_leaves_the_others_alone():
    rng = np.random.default_rng(4)
    c = marker_cache(4, 3)
    before = c.copy()
    lat, rope = _tokens(rng, 30)
    slots = rng.choice(4 * 64, 30, replace=False)
    layered.pack_into_layered_cache(lat, rope, slots, c, 1)
    assert np.array_equal(c[:, 0], before[:, 0]) and np.array_equal(c[:, 2], before[:, 2])
    ref = before[:, 1].copy()
    pack.pack_into_cache(lat, rope, slots, ref)
    assert np.array_equal(c[:, 1], ref)
    # the bytes of slot s of layer 1 sit at the layout formula
    flat = c.reshape(-1)
    for s in slots[:5]:
        off = layered.row_byte_offset(int(s) // 64, 1, int(s) % 64, 3)
        assert np.array_equal(flat[off:off + 352], ref.reshape(-1, 352)[s])


def test_layered_decode_is_the_one_layer_decode():
    rng = np.random.default_rng(5)
    nb, nl, layer = 6, 3, 2
    c = np.zeros((nb, nl, 64, 352), dtype=np.uint8)
    for l in range(nl):
        lat, rope = _tokens(rng, nb * 64)
        layered.pack_into_layered_cache(lat, rope, np.arange(nb * 64), c, l)
    T, H = 2, 4
    q_lat = rng.standard_normal((T, H, 512))
    q_rope = rng.standard_normal((T, H, 64))
    bt = rng.permutation(nb)[None, :].astype(np.int64)
    topk = np.stack([rng.choice(nb * 64, 50, replace=False) for _ in range(T)])
    o1, l1, b1 = layered.sparse_mla_decode_layered(q_lat, q_rope, c, layer, bt, topk, 0.1)
    o2, l2, b2 = oatt.sparse_mla_decode(q_lat, q_rope, np.ascontiguousarray(c[:, layer]), bt, topk, 0.1)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2) and b1 == b2 == 0
    # and another layer's rows give another answer
    o3, _, _ = layered.sparse_mla_decode_layered(q_lat, q_rope, c, 0, bt, topk, 0.1)
    assert not np.allclose(o1, o3)

"""Pins for the oracle's FP8 cache (CPU only): the 576-byte row (sizes from
the pages, tests/golden/layout.txt), values that E4M3 holds exactly come back
exactly, saturation at 448, and the decode over FP8 rows equals brute-force
dense attention over the decoded rows, and the staged path's attention over
the same rows."""
import numpy as np

import golden_io
from oracle import attention as oatt
from oracle import fp8cache, formats, staged


def test_row_layout():
    L = golden_io.layout()
    row = fp8cache.pack_rows(np.zeros((1, 512)), np.zeros((1, 64)))
    assert row.shape == (1, L["row_bytes_fp8"]) == (1, L["latent_values"] + L["rope_values"])


def test_exact_values_round_trip():
    rng = np.random.default_rng(0)
    vals = formats.e4m3_decode(rng.integers(0, 256, (20, 576)))
    vals[np.isnan(vals)] = 0.0
    row = fp8cache.pack_rows(vals[:, :512], vals[:, 512:])
    lat, rope = fp8cache.unpack_rows(row)
    assert np.array_equal(lat, vals[:, :512]) and np.array_equal(rope, vals[:, 512:])


def test_saturation():
    row = fp8cache.pack_rows(np.full((1, 512), 1e6), np.full((1, 64), -1e6))
    lat, rope = fp8cache.unpack_rows(row)
    assert (lat == 448).all() and (rope == -448).all()


def test_decode_is_dense_attention_and_matches_the_staged_attention():
    rng = np.random.default_rng(1)
    n, T, H = 256, 2, 4
    lat = rng.standard_normal((n, 512))
    rope = rng.standard_normal((n, 64))
    cache = np.zeros((n // 64, 64, 576), dtype=np.uint8)
    fp8cache.pack_into_cache(lat, rope, np.arange(n), cache)
    q_lat = rng.standard_normal((T, H, 512))
    q_rope = rng.standard_normal((T, H, 64))
    bt = rng.permutation(n // 64)[None, :]
    topk = np.stack([rng.choice(n, 40, replace=False) for _ in range(T)])
    out, lse, bad = fp8cache.sparse_mla_decode(q_lat, q_rope, cache, bt, topk, 0.1)
    assert bad == 0
    flat = cache.reshape(-1, 576)
    for t in range(T):
        slots = bt[0, topk[t] // 64] * 64 + topk[t] % 64
        K_lat, K_rope = fp8cache.unpack_rows(flat[slots])
        s = 0.1 * (q_lat[t] @ K_lat.T + q_rope[t] @ K_rope.T)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        np.testing.assert_allclose(out[t], (p @ K_lat) / p.sum(axis=1, keepdims=True), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[t], (m[:, 0] + np.log(p.sum(axis=1))), rtol=1e-12, atol=1e-12)
        # the staged path's stage 2 reads rows in the same format
        buf = flat[slots][None]
        o2, l2 = staged.decode_fp8rows(q_lat[t:t + 1], q_rope[t:t + 1], buf, np.arange(40)[None], 0.1)
        np.testing.assert_allclose(o2[0], out[t], rtol=1e-12, atol=1e-12)

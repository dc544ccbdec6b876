"""Pins for the oracle's cache-row writer (CPU only).

The row layout is checked against the byte counts the pages print
(tests/golden/layout.txt) and against a row derived by hand
(tests/golden/hand_row.txt); the quantiser against bounds that follow from
round-to-nearest on the E2M1 grid.
"""
import numpy as np
import pytest
import torch

import golden_io
from oracle import formats, pack


def check_layout():
    L = golden_io.layout()
    assert pack.LATENT == L["latent_values"]
    assert pack.GROUP == L["group_values"]
    assert pack.ROPE == L["rope_values"]
    code_bytes = L["latent_values"] * L["bits_per_latent_value"] / 8
    scale_bytes = L["latent_values"] / L["group_values"] * L["scale_bytes_per_group"]
    rope_bytes = L["rope_values"] * L["rope_bytes_per_value"]
    assert code_bytes + scale_bytes + rope_bytes == L["row_bytes_nvfp4"] == pack.ROW_BYTES
    assert (pack.CODE_BYTES, pack.SCALE_OFF, pack.ROPE_OFF) == (code_bytes, code_bytes, code_bytes + scale_bytes)
    assert L["latent_values"] + L["rope_values"] == L["row_bytes_fp8"]
    # a packed row really is 352 bytes
    row = pack.pack_rows(np.zeros((1, 512)), np.zeros((1, 64)))
    assert row.shape == (1, L["row_bytes_nvfp4"])


def test_layout_matches_pages():
    check_layout()


def check_hand_row():
    h = golden_io.hand_row()
    # the fixture's values are exact in bf16 (the pack input type)
    bf = torch.tensor(h["latent"]).to(torch.bfloat16).double().numpy()
    assert np.array_equal(bf, h["latent"])
    got = pack.pack_rows(h["latent"][None], h["rope"][None])[0]
    assert np.array_equal(got, h["row"]), np.nonzero(got != h["row"])


def test_hand_row():
    check_hand_row()


def test_hand_row_codes_match_bytes():
    h = golden_io.hand_row()
    for g, codes in h["codes"].items():
        b = h["row"][8 * g:8 * g + 8]
        assert list(b & 15) == codes[0::2] and list(b >> 4) == codes[1::2]


def test_unpack_inverts_hand_row():
    h = golden_io.hand_row()
    lat, rope = pack.unpack_row(h["row"])
    S = formats.E4M3_TABLE[h["row"][256:288]]
    # group 0 is exactly on the grid with S = 1
    assert np.array_equal(lat[:16], h["latent"][:16])
    assert np.all(S[7:] == 0) and np.all(lat[16 * 7:] == 0)
    assert rope[0] == 1.0 and rope[1] == -2.0 and rope[4] == -448.0


def test_quantisation_error_bound():
    """Round-to-nearest on the grid: |x - q| is at most half the local grid
    step times S, except where |x| / S exceeds 6 (saturation)."""
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((64, 512)) * rng.lognormal(0, 1, 512)).to(torch.bfloat16).double().numpy()
    row = pack.pack_rows(x, np.zeros((64, 64)))
    q, _ = pack.unpack_rows(row)
    S = np.repeat(formats.E4M3_TABLE[row[:, 256:288]], 16, axis=1)
    y = np.abs(x) / S
    step = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
    bound = np.where(y > 6, np.abs(x) - 6 * S, step / 2 * S)
    assert np.all(np.abs(x - q) <= bound * (1 + 1e-12))
    # with a normal (not subnormal) scale, rounding amax/6 to 3 mantissa
    # bits moves it by at most 1/17, so amax/S stays below 6 * 17/16
    amax = np.abs(x).reshape(64, 32, 16).max(-1)
    Sg = formats.E4M3_TABLE[row[:, 256:288]]
    normal = Sg >= 2.0 ** -6
    assert normal.sum() > 1000
    assert np.all(amax[normal] / Sg[normal] <= 6 * 17 / 16)


def test_pack_into_cache_addressing():
    rng = np.random.default_rng(1)
    lat = rng.standard_normal((5, 512))
    rope = rng.standard_normal((5, 64))
    cache = np.zeros((3, 64, 352), dtype=np.uint8)
    slots = np.array([0, 63, 64, -1, 191])
    pack.pack_into_cache(lat, rope, slots, cache)
    rows = pack.pack_rows(lat, rope)
    assert np.array_equal(cache[0, 0], rows[0])
    assert np.array_equal(cache[0, 63], rows[1])
    assert np.array_equal(cache[1, 0], rows[2])
    assert np.array_equal(cache[2, 63], rows[4])
    assert int(np.count_nonzero(cache.reshape(-1, 352).any(axis=1))) == 4
    with pytest.raises(IndexError):
        pack.pack_into_cache(lat[:1], rope[:1], np.array([192]), cache)

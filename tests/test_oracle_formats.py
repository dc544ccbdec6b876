"""Pins for the oracle's number formats (CPU only).

Each check compares the oracle with something other than itself: the E2M1
grid the pages' format fixes (tests/golden/layout.txt), torch's float8_e4m3fn
conversion (a library routine), and a textbook round-half-even restatement
of FP4/FP8 rounding written with numpy.rint.
"""
import numpy as np
import pytest
import torch

import golden_io
from oracle import formats

ALL_BF16 = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
FINITE_BF16 = ALL_BF16[torch.isfinite(ALL_BF16)].double().numpy()


def torch_e4m3(x):
    """torch's float8_e4m3fn code of float64 values (RNE; NaN beyond 464)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def textbook_rne(y, mant_bits, min_exp, max_val):
    """Round |y| (float64, exact inputs) to a binary format with `mant_bits`
    stored mantissa bits, smallest normal exponent `min_exp`, saturating at
    max_val, using numpy's round-half-even on the scaled value."""
    y = np.abs(np.asarray(y, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(y > 0, y, 1.0)))
    e = np.maximum(e, min_exp)
    q = 2.0 ** (e - mant_bits)
    r = np.rint(y / q) * q
    return np.minimum(r, max_val)


def check_e2m1_grid():
    grid = np.array(golden_io.layout()["e2m1_grid"])
    t = formats.E2M1_TABLE
    assert np.array_equal(t[:8], grid)
    assert np.array_equal(t[8:], -grid)
    assert np.signbit(t[8]) and not np.signbit(t[0])


def test_e2m1_table_is_the_grid():
    check_e2m1_grid()


def test_e4m3_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    ours = formats.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_named_values():
    assert formats.e4m3_value(0x38) == 1.0
    assert formats.e4m3_value(0x7E) == 448.0
    assert formats.e4m3_value(0x01) == 2.0 ** -9
    assert formats.e4m3_value(0x08) == 2.0 ** -6
    assert formats.e4m3_value(0xC0) == -2.0


def check_e4m3_encode_all_bf16():
    x = FINITE_BF16
    ours = formats.e4m3_encode(x)
    inr = np.abs(x) < 448.0
    assert np.array_equal(ours[inr], torch_e4m3(x[inr]))
    sat = ~inr
    assert np.all(ours[sat] == np.where(x[sat] < 0, 0xFE, 0x7E))
    # textbook restatement of the magnitudes
    mag = formats.E4M3_TABLE[ours & 0x7F]
    assert np.array_equal(mag, textbook_rne(x, 3, -6, 448.0))


def test_e4m3_encode_all_bf16():
    check_e4m3_encode_all_bf16()


def check_scale_encode_all_bf16():
    amax = FINITE_BF16[~np.signbit(FINITE_BF16)]
    ours = formats.e4m3_encode_quotient(amax, 6.0)
    # library: fp32 quotient (correctly rounded) then torch's RNE cast; the
    # quotient of an 8-bit value by 6 never lands on an FP8 tie by rounding
    q32 = (amax.astype(np.float32) / np.float32(6.0))
    inr = q32 < 448.0
    assert np.array_equal(ours[inr], torch_e4m3(q32[inr]))
    assert np.all(ours[~inr] == 0x7E)
    assert np.array_equal(formats.E4M3_TABLE[ours], textbook_rne(amax / 6.0, 3, -6, 448.0))


def test_scale_encode_all_bf16():
    check_scale_encode_all_bf16()


E2M1_CODE_OF = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def textbook_e2m1(y):
    """E2M1 rounding of |y| by binade: step 0.5 below 2, 1 below 4, 2 above,
    numpy round-half-even, saturating at 6."""
    y = np.abs(y)
    r = np.where(y < 2, np.rint(2 * y) / 2, np.where(y < 4, np.rint(y), 2 * np.rint(y / 2)))
    return np.minimum(r, 6.0)


def check_e2m1_encode_exhaustive():
    x = FINITE_BF16
    scales = formats.E4M3_TABLE[1:127]  # every non-zero finite scale
    rng = np.random.default_rng(0)
    huge = x[np.abs(x) > 1e30]
    for S in scales:
        # values in the range that matters for this scale, random others from
        # the whole bf16 range, and the largest magnitudes (saturation)
        xs = np.concatenate([x[(np.abs(x) <= 8 * S) & (np.abs(x) >= S / 8)], rng.choice(x, 256),
                             rng.choice(huge, 64)])
        codes = formats.e2m1_encode_scaled(xs, S)
        ref = textbook_e2m1(xs / S)
        got = formats.E2M1_TABLE[codes & 7]
        assert np.array_equal(got, ref), S
        assert np.array_equal(codes >> 3, np.signbit(xs).astype(np.uint8))


def test_e2m1_encode_exhaustive():
    check_e2m1_encode_exhaustive()


def test_e2m1_zero_scale_keeps_only_signs():
    x = np.array([0.0, -0.0, 1.0, -3.0, 1e-30])
    assert list(formats.e2m1_encode_scaled(x, 0.0)) == [0, 8, 0, 8, 0]


def test_on_grid_round_trip():
    for S in formats.E4M3_TABLE[1:127]:
        for c in range(16):
            v = formats.E2M1_TABLE[c] * S
            got = formats.e2m1_encode_scaled(np.array([v]), S)[0]
            assert formats.E2M1_TABLE[got] * S == v


def test_encoders_reject_non_finite():
    with pytest.raises(ValueError):
        formats.e4m3_encode([np.nan])
    with pytest.raises(ValueError):
        formats.e2m1_encode_scaled([np.inf], 1.0)

"""Oracle: the two number formats of an NVFP4 cache row (TEST INFRASTRUCTURE).

"Prime Inference: Fast, Reliable Serving for Frontier Open Models", section
"Making room for low-latency decode": the 512-value latent is stored in NVFP4,
four bits per value with one FP8 scale per group of 16 values, and the
64-value positional part stays FP8.

* FP4 is E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. Its
  magnitudes are {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* FP8 is E4M3 in its "FN" form: 1 sign bit, 4 exponent bits (bias 7),
  3 mantissa bits, subnormals at exponent field 0, no infinities, and the
  all-ones pattern S.1111.111 is NaN, so the largest finite value is 448.

Encoding is round-to-nearest, ties to the code with even mantissa (even code
index among the non-negative codes), saturating to the largest finite value;
the sign bit is copied from the input, so values that round to zero keep
their sign (-0 encodes as the negative-zero code).

All arithmetic is float64. The encoders pick the nearest table entry by
comparing exact distances; the tables are built from the bit-field definitions
above, not from any hardware routine.
"""
from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (sign in bit 3)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = 0.5 * m  # subnormal: m/2 * 2^(1-1)
    else:
        mag = (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -mag if s else mag


def e4m3_value(code: int) -> float:
    """Value of an 8-bit E4M3 (FN) code; NaN for S.1111.111."""
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
# non-negative finite codes 0..126, ascending in value
_E4M3_POS = E4M3_TABLE[:127].copy()
_E2M1_POS = E2M1_TABLE[:8].copy()


_CHUNK = 1 << 16


def _chunked(fn, *arrays):
    """Apply fn to matching flat chunks of equally shaped arrays (bounds the
    size of the candidate-distance matrices; no effect on the result)."""
    shape = arrays[0].shape
    flat = [np.ascontiguousarray(a).reshape(-1) for a in arrays]
    out = np.empty(flat[0].size, dtype=np.uint8)
    for i in range(0, out.size, _CHUNK):
        out[i:i + _CHUNK] = fn(*[f[i:i + _CHUNK] for f in flat])
    return out.reshape(shape)


def _nearest_even(dist: np.ndarray) -> np.ndarray:
    """Index of the smallest distance along the last axis; among equal
    smallest distances the even index wins (the candidates are consecutive
    codes, so an exact tie is always between one even and one odd code)."""
    best = dist.min(axis=-1, keepdims=True)
    hit = dist == best
    idx = np.arange(dist.shape[-1])
    # prefer even indices: score = index, minus a large bonus for even ones
    score = np.where(hit, np.where(idx % 2 == 0, idx - 10_000, idx), 1 << 30)
    return score.argmin(axis=-1)


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even, saturating E4M3 code (uint8) of each value.

    Values whose magnitude exceeds 448 become 448. The nearest table entry is
    found by comparing |x| with every finite non-negative E4M3 value."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("e4m3_encode: inputs must be finite")
    def one(xc):
        a = np.abs(xc)
        dist = np.abs(a[:, None] - _E4M3_POS)
        code = _nearest_even(dist).astype(np.uint8)
        code = np.where(a >= E4M3_MAX, np.uint8(126), code).astype(np.uint8)
        return code | np.where(np.signbit(xc), np.uint8(0x80), np.uint8(0))

    return _chunked(one, x)


def e4m3_encode_quotient(num, den: float) -> np.ndarray:
    """E4M3 code of the real quotient num/den for num >= 0, den > 0, rounded
    to nearest even and saturated, without dividing: the nearest table value
    e minimises |num - den*e|. With num a bf16 value and den*e holding at
    most 6 significant bits, these differences are exact in float64 whenever
    they can tie."""
    num = np.asarray(num, dtype=np.float64)
    if np.any(num < 0) or not np.all(np.isfinite(num)):
        raise ValueError("e4m3_encode_quotient: numerators must be finite and >= 0")
    def one(nc):
        dist = np.abs(nc[:, None] - den * _E4M3_POS)
        code = _nearest_even(dist).astype(np.uint8)
        return np.where(nc >= den * E4M3_MAX, np.uint8(126), code)

    return _chunked(one, num)


def e2m1_encode_scaled(x, scale) -> np.ndarray:
    """4-bit E2M1 code of x / scale, round-to-nearest-even, saturating at 6.

    ``scale`` is the decoded (already rounded) group scale and broadcasts
    against x. The nearest grid point g minimises |x| - g*scale| (exact in
    float64: g*scale has at most 6 significant bits); |x| >= 6*scale gives
    the largest magnitude. A zero scale gives
    magnitude code 0 for every value. The sign bit is copied from x."""
    x = np.asarray(x, dtype=np.float64)
    scale = np.broadcast_to(np.asarray(scale, dtype=np.float64), x.shape)
    if not np.all(np.isfinite(x)):
        raise ValueError("e2m1_encode_scaled: inputs must be finite")
    def one(xc, sc):
        a = np.abs(xc)
        dist = np.abs(a[:, None] - sc[:, None] * _E2M1_POS)
        mag = _nearest_even(dist).astype(np.uint8)
        # saturation: at or beyond 6*S the largest magnitude is the answer
        # (stated explicitly: far beyond 6*S the float64 distances to the
        # grid points are all rounded to |x| and can no longer tell)
        mag = np.where(a >= E2M1_MAX * sc, np.uint8(7), mag)
        mag = np.where(sc == 0.0, np.uint8(0), mag).astype(np.uint8)
        return mag | np.where(np.signbit(xc), np.uint8(8), np.uint8(0))

    return _chunked(one, x, np.ascontiguousarray(scale))


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.int64) & 15]


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.int64) & 255]

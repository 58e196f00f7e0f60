"""Number formats used by the compressed cache, from their definitions (oracle).

TEST INFRASTRUCTURE ONLY.  Part of the CPU oracle; the product path never
imports it.

FP8-E4M3 (the metadata format the ResidualQuant pages name: "FP8 scale and
offset" per channel group, ai4snews summary, main-results paragraph):
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
the all-ones pattern (S.1111.111) is NaN.  Subnormals: m * 2^-9 for m in
1..7.  Normals: (1 + m/8) * 2^(e-7), e in 1..15.  Largest finite 448.

BF16 (the format of the per-vector least-squares coefficient: "BF16
least-squares coefficient", same paragraph): 1 sign, 8 exponent bits with
bias 127, 7 mantissa bits; the top half of an IEEE binary32.

Rounding is round-to-nearest, ties to the even significand, applied to the
exact value of a float64 argument.  E4M3 saturates: magnitudes past 448 go
to 448 (the "satfinite" reading; the pages do not say, and it is the only
choice that never stores NaN metadata).
"""
from __future__ import annotations

import numpy as np

__all__ = ["E4M3_MAX", "e4m3_encode", "e4m3_decode", "e4m3_round",
           "bf16_encode", "bf16_decode", "bf16_round", "e4m3_all_finite", "fma_f32"]

E4M3_MAX = 448.0
_E4M3_MIN_NORMAL_EXP = -6   # smallest normal 2^-6
_E4M3_SUBNORMAL_QUANTUM = 2.0 ** -9
_E4M3_MANT_BITS = 3

_BF16_MIN_NORMAL_EXP = -126
_BF16_SUBNORMAL_QUANTUM = 2.0 ** -133
_BF16_MANT_BITS = 7


def _round_to_format(x: np.ndarray, mant_bits: int, min_normal_exp: int,
                     sub_quantum: float) -> np.ndarray:
    """Round float64 values to a binary format with `mant_bits` stored mantissa bits.

    The spacing (quantum) of representable numbers in the binade
    [2^e, 2^(e+1)) is 2^(e - mant_bits); below the smallest normal it is the
    subnormal quantum.  Dividing by the quantum (a power of two, so exact)
    gives a real k; np.rint takes the nearest integer with ties to even, and
    an even k is an even significand.  k * quantum is the rounded value.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e2 = np.frexp(ax)              # ax = f * 2^e2, f in [0.5, 1)
    e = e2.astype(np.int64) - 1       # ax in [2^e, 2^(e+1))
    e = np.maximum(e, min_normal_exp)
    quantum = np.where(ax < 2.0 ** min_normal_exp, sub_quantum,
                       np.ldexp(1.0, (e - mant_bits).astype(np.int32)))
    k = np.rint(ax / quantum)
    return np.copysign(k * quantum, x)


def e4m3_round(x) -> np.ndarray:
    """Value of x rounded to E4M3 (RNE, saturating at +-448), as float64."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no E4M3 metadata encoding in this cache format")
    r = _round_to_format(np.clip(x, -E4M3_MAX, E4M3_MAX), _E4M3_MANT_BITS,
                         _E4M3_MIN_NORMAL_EXP, _E4M3_SUBNORMAL_QUANTUM)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def e4m3_all_finite():
    """(codes 0..126, magnitudes) of the non-negative finite E4M3 values, increasing."""
    codes = np.arange(0x7F, dtype=np.uint8)
    return codes, e4m3_decode(codes)


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 byte (NaN for the NaN pattern)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * _E4M3_SUBNORMAL_QUANTUM,
                   (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int32)))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """E4M3 byte of round(x) (RNE, saturating).  The sign bit follows the sign of x,
    so a negative value that rounds to zero is stored as 0x80 (negative zero)."""
    x = np.asarray(x, dtype=np.float64)
    r = e4m3_round(x)
    ar = np.abs(r)
    _, e2 = np.frexp(ar)
    e_unb = e2.astype(np.int64) - 1
    is_sub = ar < 2.0 ** _E4M3_MIN_NORMAL_EXP
    sub_m = np.rint(ar / _E4M3_SUBNORMAL_QUANTUM).astype(np.int64)
    norm_e = np.clip(e_unb + 7, 1, 15)
    frac = ar / np.ldexp(1.0, e_unb.astype(np.int32)) - 1.0
    norm_m = np.rint(frac * 8.0).astype(np.int64)
    mag = np.where(is_sub, sub_m, (norm_e << 3) | norm_m)
    neg = np.signbit(x)
    return (mag | np.where(neg, 0x80, 0)).astype(np.uint8)


def bf16_round(x) -> np.ndarray:
    """Value of x rounded to BF16 (RNE), as float64.  Inputs here are finite and
    within range (no overflow handling needed for the cache's coefficients)."""
    x = np.asarray(x, dtype=np.float64)
    return _round_to_format(x, _BF16_MANT_BITS, _BF16_MIN_NORMAL_EXP, _BF16_SUBNORMAL_QUANTUM)


def bf16_encode(x) -> np.ndarray:
    """uint16 bit pattern of round(x) in BF16 (the value is exact in binary32,
    whose top half it is)."""
    r = bf16_round(x).astype(np.float32)  # exact: every BF16 value is a binary32 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def bf16_decode(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _round_to_odd_sum(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a + b rounded to float64 with round-to-odd: the exact sum if representable,
    else whichever neighbouring float64 has an odd significand (TwoSum gives the
    exact rounding error of the nearest-even sum)."""
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)
    odd = (s.view(np.uint64) & np.uint64(1)).astype(bool)
    toward = np.where(err > 0, np.inf, -np.inf)
    return np.where((err == 0) | odd, s, np.nextafter(s, toward))


def fma_f32(a, b, c) -> np.ndarray:
    """IEEE binary32 fused multiply-add round(a*b + c), nearest-even, one rounding.

    a, b, c must hold binary32 values (any float dtype).  a*b is exact in
    float64 (24 + 24 bits); adding c with round-to-odd keeps a sticky bit, so
    the final cast to float32 rounds exactly once (float64 carries more than
    two bits beyond binary32's 24)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    p = a * b
    return _round_to_odd_sum(p, np.broadcast_to(c, p.shape).astype(np.float64)).astype(np.float32)

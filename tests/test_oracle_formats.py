"""Pins for the oracle's E4M3 and BF16 rounding (no GPU).

Each check ties the oracle to something other than itself: a library cast
(torch's float8_e4m3fn / bfloat16), exact rational arithmetic (fractions),
or values fixed by the format definitions.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F


def _e4m3_table():
    """All finite non-negative E4M3 values from torch's own decoder."""
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    return codes.numpy(), codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_on_all_bytes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.e4m3_decode(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])


@pytest.mark.parametrize("x,code", [
    (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (2.0 ** -9, 0x01), (7 * 2.0 ** -9, 0x07),
    (2.0 ** -6, 0x08), (0.0, 0x00), (1.0625, 0x38), (1.1875, 0x3A), (0.5 * 2.0 ** -9, 0x00),
    (1.5 * 2.0 ** -9, 0x02), (500.0, 0x7E), (-1000.0, 0xFE), (240.0, 0x77), (0.3, 0x2A),
])
def test_e4m3_fixed_points(x, code):
    # 1.0625 lies halfway between 1.0 (m=0) and 1.125 (m=1): ties go to the even m.
    # 1.1875 lies halfway between 1.125 (m=1) and 1.25 (m=2): goes to m=2.
    assert int(F.e4m3_encode(x)) == code


def test_e4m3_negative_underflow_keeps_sign():
    assert int(F.e4m3_encode(-1e-30)) == 0x80
    assert int(F.e4m3_encode(-0.0)) == 0x80


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 3,
        rng.standard_normal(20000) * 0.01, rng.uniform(-2 ** -6, 2 ** -6, 5000),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.e4m3_encode(x.astype(np.float64))
    # torch keeps the sign of values that round to zero too
    assert np.array_equal(ref, ours)


def test_e4m3_midpoints_brute_force():
    """Every midpoint between neighbouring finite values, +-1 ulp of float64,
    rounds as exact nearest-even says (Fraction arithmetic)."""
    codes, vals = _e4m3_table()
    for i in range(len(vals) - 1):
        lo, hi = Fraction(vals[i]), Fraction(vals[i + 1])
        mid = (lo + hi) / 2
        for x in (float(mid), np.nextafter(float(mid), -np.inf), np.nextafter(float(mid), np.inf)):
            fx = Fraction(x)
            if abs(fx - lo) < abs(hi - fx):
                want = codes[i]
            elif abs(fx - lo) > abs(hi - fx):
                want = codes[i + 1]
            else:
                want = codes[i] if codes[i] % 2 == 0 else codes[i + 1]
            assert int(F.e4m3_encode(x)) == int(want), (x, vals[i], vals[i + 1])


def test_bf16_matches_torch_cast_from_fp32():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(50000), rng.uniform(-1e3, 1e3, 5000),
                        rng.standard_normal(5000) * 1e-30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.bf16_encode(x.astype(np.float64)), ref)
    assert np.array_equal(F.bf16_decode(ref), torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_bf16_rounds_float64_exactly():
    """float64 inputs that fall between float32 values: exact nearest-even (no
    double rounding through float32)."""
    rng = np.random.default_rng(3)
    for _ in range(2000):
        base = np.float32(rng.uniform(0.5, 2.0))
        bits = int(torch.tensor(base).to(torch.bfloat16).view(torch.int16)) & 0xFFFF
        lo = float(torch.tensor(bits, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double())
        hi = float(torch.tensor(bits + 1, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double())
        mid = (lo + hi) / 2
        for x in (mid - 1e-12, mid + 1e-12, mid, np.nextafter(mid, 0.0), np.nextafter(mid, 9.0)):
            fx = Fraction(x)
            dl, dh = abs(fx - Fraction(lo)), abs(Fraction(hi) - fx)
            got = float(F.bf16_round(x))
            if dl < dh:
                assert got == lo
            elif dh < dl:
                assert got == hi
            else:
                assert got == (lo if bits % 2 == 0 else hi)

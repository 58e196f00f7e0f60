"""The hand-built edge vectors (tests/edge_inputs.py) reach the edges they aim at.

CPU only.  Each pattern is run through the oracle's group compression and the
stored bytes are compared with values worked out by hand from the quantizer's
definition (offset o = E4M3(min), scale s = E4M3(range / (2^b - 1)), nearest
grid point with ties to even, s = 0 giving code 0: the worked storage example
of the explainer and the main-results paragraph of the ai4snews summary).
So the GPU edge-case tests cannot pass without exercising those edges, and
these checks double as oracle pins at the edges.
"""
import numpy as np
import pytest

import oracle
import synth
from edge_inputs import ALL_KINDS, check_bf16_exact, edge_kv, pattern

E4M3_448, E4M3_NEG_448, E4M3_NEG_ZERO = 0x7E, 0xFE, 0x80


def _compress(kind, d=128, g=32, P=4, seed=0, R=None):
    x = pattern(kind, np.random.default_rng(seed), d, g, P)
    check_bf16_exact(x)
    R = synth.rotation(d).astype(np.float32).astype(np.float64) if R is None else R
    return x, oracle.compress_group(x, R, g)


@pytest.mark.parametrize("d,g", [(128, 32), (96, 16)])
def test_const_group_stores_zero_scale_and_zero_codes(d, g):
    x, c = _compress("const_group", d, g)
    codes, s, o = c["anchor"]
    assert s[0] == 0 and not codes[:g].any()
    assert oracle.e4m3_decode(o[:1])[0] == 1.5


@pytest.mark.parametrize("d,g", [(128, 32), (96, 32)])
def test_zero_residual_is_exact(d, g):
    x, c = _compress("zero_residual", d, g)
    for j in range(3):
        rc, rs, ro, cb = c["res"][j]
        assert oracle.bf16_decode(np.array([cb]))[0] == 0.75
        assert not rc.any() and not rs.any() and not ro.any()
        assert np.array_equal(c["recon"][j], x[j])
    assert np.array_equal(c["recon"][3], x[3])   # the anchor sits on its own grid


def test_zero_anchor_gives_zero_coefficient():
    x, c = _compress("zero_anchor")
    codes, s, o = c["anchor"]
    assert not codes.any() and not s.any() and not o.any()
    for j in range(3):
        assert c["res"][j][3] == 0   # c = 0: BF16 bits 0x0000


def test_subnormal_scale_and_offset():
    x, c = _compress("subnormal")
    codes, s, o = c["anchor"]
    assert s[0] == 0x01                       # 2^-9, the smallest E4M3 subnormal
    assert o[1] == 0x03 and s[1] == 0x00      # offset 3 x 2^-9; scale rounds to 0
    assert np.array_equal(codes[:32], np.rint((x[3, :32] - 1.0) / 2.0 ** -9).astype(np.uint8))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_ties_go_to_the_even_code(seed):
    x, c = _compress("ties", seed=seed)
    codes = c["anchor"][0]
    a = x[3]
    # group 0: o = 0, s = 1/4; group 1: o = -2, s = 1/2 (exact, by the pattern's ends)
    t0 = a[:32] / 0.25
    t1 = (a[32:64] + 2.0) / 0.5
    assert np.sum(t0 % 1 == 0.5) >= 20 and np.sum(t1 % 1 == 0.5) >= 20   # most are exact ties
    # np.rint rounds halves to even: the textbook rule, computed independently
    assert np.array_equal(codes[:32], np.rint(t0).astype(np.uint8))
    assert np.array_equal(codes[32:64], np.rint(t1).astype(np.uint8))


def test_negative_tiny_minimum_gives_negative_zero_offset():
    x, c = _compress("neg_zero_offset")
    assert c["anchor"][2][0] == E4M3_NEG_ZERO


@pytest.mark.parametrize("d", [128, 96])
def test_coefficient_on_and_above_bf16_midpoints(d):
    x, c = _compress("c_midpoint", d=d, g=32)
    # all-ones anchor: every group constant, offset 1, codes 0
    assert not c["anchor"][0].any() and not c["anchor"][1].any()
    bits = [c["res"][j][3] for j in range(3)]
    assert bits == [0x3F80, 0x3F81, 0x3F82]   # 1 (tie to even), 1 + 2^-7 (above), 1 + 2^-6 (tie to even)


def test_saturation_of_offset_and_scale():
    x, c = _compress("saturation")
    assert c["anchor"][2][0] == E4M3_NEG_448 and c["anchor"][1][0] == E4M3_448


def test_edge_kv_places_every_kind():
    rng = np.random.default_rng(3)
    kv = edge_kv(rng, list(ALL_KINDS), 4, 2, 3, 9, 128, 32)
    assert kv.shape == (4, 2, 2, 3, 9, 128)
    # token (b=0, h=0, t=1) of K got the second kind, the zero residual: loops 0.75 x anchor
    assert np.array_equal(kv[0, 0, 0, 0, 1], 0.75 * kv[3, 0, 0, 0, 1])

"""Hand-built K/V vectors that reach the edges of the ResidualQuant quantizer.

Inputs only: every vector here is written down directly (values on a known
grid, constant runs, exact ties) and rounded to nothing -- each value is
exactly representable in BF16 by construction, and `check_bf16_exact`
asserts it.  None of the compression arithmetic lives here; which edge a
pattern reaches is pinned separately by running the oracle on it
(tests/test_edge_inputs.py).

A pattern is a float64 array [P, d] for one (K or V) vector of one token:
index P-1 is the group's last loop (the INT4 anchor), indices 0..P-2 the
earlier loops (2-bit residuals).  The group quantizer stores, per channel
group, offset o = E4M3(min) and scale s = E4M3((max - min) / (2^b - 1)) (the
explainer's worked storage example; the ai4snews summary's main-results
paragraph, FP8 scale and offset); the patterns aim at its special cases:

  const_group      one anchor channel group constant: s = 0, every code 0
  zero_residual    anchor on the INT4 grid with E4M3-exact o and s, every
                   earlier loop 0.75 x anchor: c = 0.75 exactly, residual 0
  zero_anchor      anchor all zero: o = s = 0, c = 0, the residual is the loop
  subnormal        a group whose range / 15 is an E4M3 subnormal; a group whose
                   offset is an E4M3 subnormal and whose scale rounds to 0
  ties             values exactly halfway between grid points o + k s (ties
                   go to the even k)
  neg_zero_offset  a group minimum that rounds to E4M3 -0 (offset byte 0x80)
  c_midpoint       all-ones anchor; loops whose least-squares coefficient is a
                   BF16 midpoint (tie to even), or just above one
  saturation       a group with min < -448 and range > 448 x 15 (E4M3 offset
                   and scale both saturate)
"""
from __future__ import annotations

import numpy as np

KINDS_O1 = ("const_group", "zero_residual", "zero_anchor", "subnormal", "ties", "neg_zero_offset",
            "c_midpoint")
ALL_KINDS = KINDS_O1 + ("saturation",)


def check_bf16_exact(x: np.ndarray) -> None:
    """Every value of x is a BF16 number (the top 16 bits of its binary32 form)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64)), "not binary32-exact"
    bits = f.view(np.uint32)
    assert not np.any(bits & np.uint32(0xFFFF)), "not BF16-exact"


def _bf16_normal(rng: np.random.Generator, shape, scale=1.0) -> np.ndarray:
    """Gaussian values truncated to BF16 (drop the low 16 bits of binary32)."""
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (f.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)


def _loops_near(rng, a, P):
    """Earlier loops near the anchor: 0.875 x anchor plus small BF16 noise."""
    out = np.empty((P, a.size))
    out[P - 1] = a
    for l in range(P - 1):
        out[l] = 0.875 * a + _bf16_normal(rng, a.size, 0.25)
        out[l] = (out[l].astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    return out


def _grid_group(rng, o, s, g, kmin=0, kmax=15):
    """g values o + k s with k in [kmin, kmax], both ends present."""
    k = rng.integers(kmin, kmax + 1, g)
    k[0], k[1] = kmin, kmax
    rng.shuffle(k)
    return o + k * s


def pattern(kind: str, rng: np.random.Generator, d: int, g: int, P: int) -> np.ndarray:
    """One [P, d] vector pair (loops x channels) reaching the edge `kind`."""
    ng = d // g
    if kind == "const_group":
        a = _bf16_normal(rng, d)
        a[:g] = 1.5
        return _loops_near(rng, a, P)
    if kind == "zero_residual":
        a = np.concatenate([_grid_group(rng, -1.0 + 0.25 * (gi % 3), 0.125, g) for gi in range(ng)])
        out = np.empty((P, d))
        out[P - 1] = a
        out[: P - 1] = 0.75 * a
        return out
    if kind == "zero_anchor":
        out = _bf16_normal(rng, (P, d))
        out[P - 1] = 0.0
        return out
    if kind == "subnormal":
        a = _bf16_normal(rng, d)
        # group 0: range 3 * 2^-7, so range / 15 = 0.0015625, between E4M3's 2^-10 and 2^-9 steps
        a[:g] = 1.0 + rng.integers(0, 4, g) * 2.0 ** -7
        a[0], a[1] = 1.0, 1.0 + 3 * 2.0 ** -7
        # group 1: minimum 0.0050048828125 (a BF16 value) rounds to the subnormal 3 x 2^-9;
        # its range is below half an E4M3 step, so the scale rounds to 0
        tiny = np.array([0.0050048828125, 0.00543212890625, 0.005859375])
        a[g:2 * g] = tiny[rng.integers(0, 3, g)]
        a[g] = tiny[0]
        return _loops_near(rng, a, P)
    if kind == "ties":
        a = _bf16_normal(rng, d)
        # group 0: o = 0, s = 0.25 (values 0 and 3.75 present); the rest on half steps
        grp = 0.25 * rng.integers(0, 15, g) + 0.125
        grp[0], grp[1] = 0.0, 3.75
        a[:g] = grp
        # group 1: o = -2, s = 0.5 (values -2 and 5.5 present); the rest on half steps
        grp = -2.0 + 0.5 * rng.integers(0, 15, g) + 0.25
        grp[0], grp[1] = -2.0, 5.5
        a[g:2 * g] = grp
        return _loops_near(rng, a, P)
    if kind == "neg_zero_offset":
        a = _bf16_normal(rng, d)
        grp = 0.5 * rng.random(g)
        grp = (grp.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
        grp[0] = -9.965896606445312e-05   # -1e-4 truncated to BF16: rounds to E4M3 -0
        grp[1] = 0.5
        a[:g] = grp
        return _loops_near(rng, a, P)
    if kind == "c_midpoint":
        out = np.ones((P, d))
        for l in range(P - 1):
            v = l % 3
            if v == 0:     # c = 1 + 2^-8: halfway between BF16 1 and 1 + 2^-7, ties to 1
                out[l, 5] = 1.0 + d / 256
            elif v == 1:   # c = 1 + 2^-8 + 2^-7 / d: just above that midpoint, rounds up
                out[l, 5] = 1.0 + d / 256
                out[l, 9] = 1.0 + 2.0 ** -7
            else:          # c = 1 + 3 x 2^-8: halfway between 1 + 2^-7 and 1 + 2^-6, ties to 1 + 2^-6
                out[l, 5] = 1.0 + 3 * d / 256
        return out
    if kind == "saturation":
        a = _bf16_normal(rng, d)
        grp = 64.0 * rng.integers(-9, 112, g)
        grp[0], grp[1] = -600.0, 7168.0
        a[:g] = grp
        return _loops_near(rng, a, P)
    raise ValueError(kind)


def edge_kv(rng: np.random.Generator, kinds, P: int, B: int, H: int, n: int, d: int, g: int,
            base: np.ndarray | None = None) -> np.ndarray:
    """float64 [P, 2, B, H, n, d]: token (b, h, t) of K (kv = 0) or V (kv = 1) gets
    pattern kinds[(t + 3 h + 5 b + kv) % len(kinds)]; a kind of None keeps `base`
    (or zeros) there."""
    out = np.zeros((P, 2, B, H, n, d)) if base is None else np.array(base, dtype=np.float64)
    for kv in range(2):
        for b in range(B):
            for h in range(H):
                for t in range(n):
                    k = kinds[(t + 3 * h + 5 * b + kv) % len(kinds)]
                    if k is not None:
                        out[:, kv, b, h, t] = pattern(k, rng, d, g, P)
    check_bf16_exact(out)
    return out


def to_bf16_tensor(x: np.ndarray):
    """The BF16 tensor holding exactly the values of x (which must be BF16-exact)."""
    import torch
    check_bf16_exact(x)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


RESIDUAL_KINDS = ("ties", "const", "subnormal", "neg_zero_offset", "saturation", None)


def residual_group(kind, rng: np.random.Generator, g: int) -> np.ndarray:
    """g values for one channel group of a rotated residual (2-bit codes, 3 steps),
    reaching the edge `kind` (None: BF16 Gaussian values)."""
    if kind == "ties":          # o = 0, s = 1; the rest exactly halfway between codes
        v = rng.integers(0, 3, g) + 0.5
        v[0], v[1] = 0.0, 3.0
    elif kind == "const":       # s = 0
        v = np.full(g, 0.6875)
    elif kind == "subnormal":   # range / 3 = 2^-9, the smallest E4M3 subnormal
        v = 0.25 + rng.integers(0, 4, g) * 2.0 ** -9
        v[0], v[1] = 0.25, 0.25 + 3 * 2.0 ** -9
    elif kind == "neg_zero_offset":
        v = rng.integers(0, 13, g) / 16.0
        v[0], v[1] = -9.965896606445312e-05, 0.75
    elif kind == "saturation":  # min < -448, range / 3 > 448
        v = 32.0 * rng.integers(-18, 64, g)
        v[0], v[1] = -600.0, 2048.0
    else:
        v = _bf16_normal(rng, g)
    rng.shuffle(v)
    return v

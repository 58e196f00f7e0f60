"""GPU: the quantizer's and the attention's edge cases, against the oracle.

The random synthetic data of the other parity tests never reaches the exact
fallback branches of the device quantizer (the E4M3 decisions near a
midpoint, the nearest code at an exact tie, the float64 re-sum of a BF16
coefficient on a midpoint) nor a softmax dominated by one key.  Here the
inputs are built to reach them (tests/edge_inputs.py; tests/test_edge_inputs.py
pins on the CPU that each pattern reaches its edge):

  * appends through rq_append and through the anchor-loop call's token append
    (rq_decode_attention_append), whose quantizer is a separate device code
    path: every cache byte equal to the oracle's;
  * attention over those caches: max |gpu - oracle| <= 2e-3 on O(1) data; where
    the data are not O(1) (E4M3 saturation, values past +-448) the bar is
    2e-3 times the largest |output| of the (row, head), i.e. the same relative
    precision;
  * a softmax that one key dominates, or two keys share, with queries x 8;
  * ragged lengths 1, 2, 31, 32, 33, 255 in one call.

Sources: the explainer "ResidualQuant stores looped-Transformer KV caches as
2-bit residuals" (worked storage example; temporary-buffer paragraph) and the
ai4snews summary's main-results paragraph (FP8 scale and offset, BF16
coefficient).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from edge_inputs import KINDS_O1, RESIDUAL_KINDS, edge_kv, residual_group, to_bf16_tensor
from rq_harness import Case, GpuCache, kv_for, rotation32

pytestmark = pytest.mark.gpu

ATOL = 2e-3


def _geom(case: Case):
    return oracle.Geometry(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax)


def _scaled_err(out, ref):
    """max over (row, head) of max|out - ref| / max(1, max|ref|)."""
    err = np.abs(out - ref).max(axis=-1)
    mag = np.maximum(1.0, np.abs(ref).max(axis=-1))
    return float((err / mag).max())


def _decode_all_loops(gpu, obuf, geom, R, case, seq, seed, chained, scaled=False, qmul=1.0):
    worst = 0.0
    scale = 1.0 / math.sqrt(case.d)
    for loop in range(case.P):
        qb, q = synth.queries(seed * 7 + loop, case.B, case.H, case.d)
        if qmul != 1.0:
            qb = (qb.float() * qmul).to(torch.bfloat16)
            q = qb.double().numpy()
        kvb, kv = synth.looped_kv(seed * 13 + loop, case.workload(), batch=case.B, ntok=1)
        out = gpu.decode(0, 0, loop, qb, kvb[loop, 0, :, :, 0], kvb[loop, 1, :, :, 0], seq, scale).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kv[loop, 0, :, :, 0], kv[loop, 1, :, :, 0],
                                      seq, scale, chained=chained)
        err = _scaled_err(out, ref) if scaled else float(np.abs(out - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"loop {loop}: error {err:.3e}"
    return worst


def _fill(case, kv, start):
    """The same tokens appended on the device (rq_append) and by the oracle."""
    R32, R = rotation32(case.d, kind=case.rotation)
    gpu = GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    gpu.append(0, 0, to_bf16_tensor(kv), start)
    oracle.append(obuf, geom, R, 0, 0, kv, start, chained=case.chained, scaling=case.scaling,
                  rotation=case.rotation)
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ after the append"
    return gpu, geom, obuf, R


def _fused_steps(gpu, obuf, geom, R, case, seq, kinds_per_step, seed, scaled=False):
    """Anchor-loop calls whose current token (every loop, K and V) is an edge
    pattern; the call appends it: bytes and outputs against the oracle."""
    rng = np.random.default_rng(seed)
    scale = 1.0 / math.sqrt(case.d)
    worst = 0.0
    for step, kind in enumerate(kinds_per_step):
        cur = edge_kv(rng, [kind], case.P, case.B, case.H, 1, case.d, case.g)[..., 0, :]   # [P,2,B,H,d]
        qb, q = synth.queries(seed + step, case.B, case.H, case.d)
        out = gpu.decode_append(0, 0, qb, to_bf16_tensor(cur), seq, scale).cpu().numpy()
        ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, cur, seq, scale, chained=case.chained,
                                                 scaling=case.scaling, rotation=case.rotation)
        assert ok.all()
        err = _scaled_err(out, ref) if scaled else float(np.abs(out - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"step {step} ({kind}): error {err:.3e}"
        gbuf = gpu.bytes_host()
        assert np.array_equal(gbuf, obuf), f"step {step} ({kind}): {int((gbuf != obuf).sum())} bytes differ"
        seq = seq + 1
    return worst


@pytest.mark.parametrize("d,g,chained", [(128, 32, False), (128, 16, False), (96, 32, False), (128, 32, True),
                                         (96, 16, True)])
def test_edge_vectors_append_decode_and_fused_append(d, g, chained):
    case = Case(L=1, P=4, G=1, H=2, d=d, g=g, B=2, Nmax=192, chained=chained, seed=70)
    n = 150
    _, base = kv_for(case, 71, n)
    kv = edge_kv(np.random.default_rng(72), list(KINDS_O1) + [None, None], 4, 2, 2, n, d, g, base=base)
    start = np.zeros(2, dtype=np.int64)
    gpu, geom, obuf, R = _fill(case, kv, start)
    seq = np.array([150, 97])
    worst = _decode_all_loops(gpu, obuf, geom, R, case, seq, 73, chained)
    worst_f = _fused_steps(gpu, obuf, geom, R, case, seq, list(KINDS_O1), 74)
    assert gpu.status.tolist() == [0, 0, 0, 0]
    print(f"d={d} g={g} chained={chained}: decode {worst:.2e}, fused {worst_f:.2e}; every byte equal")


@pytest.mark.parametrize("d,g", [(128, 32), (96, 16)])
def test_e4m3_saturation(d, g):
    """Groups past the E4M3 range: offset and scale saturate at -448 / 448; the
    codes clamp.  Bytes equal; attention at the same relative precision."""
    case = Case(L=1, P=4, G=1, H=2, d=d, g=g, B=2, Nmax=192, seed=75)
    n = 130
    _, base = kv_for(case, 76, n)
    kv = edge_kv(np.random.default_rng(77), ["saturation", None, None, None, None], 4, 2, 2, n, d, g, base=base)
    gpu, geom, obuf, R = _fill(case, kv, np.zeros(2, dtype=np.int64))
    seq = np.array([130, 66])
    worst = _decode_all_loops(gpu, obuf, geom, R, case, seq, 78, False, scaled=True)
    worst_f = _fused_steps(gpu, obuf, geom, R, case, seq, ["saturation", "saturation"], 79, scaled=True)
    assert gpu.status.tolist() == [0, 0, 0, 0]
    print(f"saturation d={d} g={g}: decode {worst:.2e}, fused {worst_f:.2e} (relative)")


@pytest.mark.parametrize("d,g", [(128, 32), (96, 16)])
def test_residual_edges_through_an_exact_rotation(d, g):
    """With R a signed permutation the rotation is exact and an all-zero anchor
    gives c = 0, so the rotated residual is exactly a designed vector: its groups
    hit exact ties, constant runs, a subnormal scale, the -0 offset and E4M3
    saturation.  Every byte equals the oracle's (which here does not depend on
    the precision reading: both agree exactly)."""
    rng = np.random.default_rng(80)
    perm = rng.permutation(d)
    sign = rng.choice([-1.0, 1.0], d)
    Rp = np.zeros((d, d), dtype=np.float32)
    Rp[np.arange(d), perm] = sign                      # u_i = sign_i x_{perm_i}
    case = Case(L=1, P=4, G=1, H=2, d=d, g=g, B=2, Nmax=128, seed=81)
    n, ng = 70, d // g
    kv = np.zeros((4, 2, 2, 2, n, d))
    for kvi in range(2):
        for b in range(2):
            for h in range(2):
                for t in range(n):
                    for lp in range(3):
                        u = np.concatenate([residual_group(RESIDUAL_KINDS[(gi + t + lp + kvi) % len(RESIDUAL_KINDS)],
                                                           rng, g) for gi in range(ng)])
                        x = np.empty(d)
                        x[perm] = sign * u                 # the loop whose rotated residual is u
                        kv[lp, kvi, b, h, t] = x
    gpu = GpuCache(case, Rp)
    geom = _geom(case)
    R = Rp.astype(np.float64)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    ob64 = np.zeros(geom.total_bytes, dtype=np.uint8)
    start = np.zeros(2, dtype=np.int64)
    gpu.append(0, 0, to_bf16_tensor(kv), start)
    oracle.append(obuf, geom, R, 0, 0, kv, start)
    oracle.append(ob64, geom, R, 0, 0, kv, start, precision="f64")
    assert np.array_equal(obuf, ob64)
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    # the designed edges are present in what the device stored
    codes, s, o, _ = oracle.read_plane_tokens(gbuf, geom, 0, 0, 0, 0, 0, "res", 0, n)
    assert (s == 0x7E).any() and (o == 0x80).any() and (s == 0x01).any() and (s == 0).any()
    seq = np.array([70, 41])
    worst = _decode_all_loops(gpu, obuf, geom, R, case, seq, 82, False, scaled=True)
    assert gpu.status.tolist() == [0, 0, 0, 0]
    print(f"exact-rotation residual edges d={d} g={g}: decode {worst:.2e} (relative); bytes equal")


@pytest.mark.parametrize("d,g", [(128, 32), (96, 32), (128, 16)])
def test_peaky_softmax(d, g):
    """Queries x 8 (a few keys carry the softmax); one row whose query is aligned
    with one cached key (that key takes almost all the weight) and one whose
    query points between two keys (they share it)."""
    case = Case(L=1, P=4, G=1, H=2, d=d, g=g, B=3, Nmax=320, seed=83)
    n = 300
    kvb, kv = kv_for(case, 84, n)
    gpu, geom, obuf, R = _fill(case, kv, np.zeros(3, dtype=np.int64))
    seq = np.array([300, 257, 129])
    scale = 1.0 / math.sqrt(d)
    worst = 0.0
    for loop in range(4):
        qb, q = synth.queries(85 + loop, 3, 2, d)
        q8 = (qb.float() * 8).to(torch.bfloat16)
        # row 1, head 0: aligned with key 77; row 2, head 1: between keys 10 and 100
        q8[1, 0] = (0.5 * torch.from_numpy(kv[loop, 0, 1, 0, 77])).to(torch.bfloat16)
        q8[2, 1] = (0.25 * torch.from_numpy(kv[loop, 0, 2, 1, 10] + kv[loop, 0, 2, 1, 100])).to(torch.bfloat16)
        qf = q8.double().numpy()
        cb, cur = synth.looped_kv(86 + loop, case.workload(), batch=3, ntok=1)
        out = gpu.decode(0, 0, loop, q8, cb[loop, 0, :, :, 0], cb[loop, 1, :, :, 0], seq, scale).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, qf, cur[loop, 0, :, :, 0], cur[loop, 1, :, :, 0],
                                      seq, scale)
        err = float(np.abs(out - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"loop {loop}: max abs err {err:.3e}"
    assert gpu.status.tolist() == [0, 0, 0, 0]
    print(f"peaky softmax d={d} g={g}: worst {worst:.2e}")


def test_ragged_lengths_with_edge_vectors():
    """Lengths 1, 2, 31, 32, 33 and 255 in one call (mid-word, word and tile
    edges); the fused call then appends edge tokens at those slots."""
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=6, Nmax=320, seed=87)
    n = 255
    _, base = kv_for(case, 88, n)
    kv = edge_kv(np.random.default_rng(89), list(KINDS_O1) + [None] * 7, 4, 6, 2, n, 128, 32, base=base)
    gpu, geom, obuf, R = _fill(case, kv, np.zeros(6, dtype=np.int64))
    seq = np.array([1, 2, 31, 32, 33, 255])
    worst = _decode_all_loops(gpu, obuf, geom, R, case, seq, 90, False)
    worst_f = _fused_steps(gpu, obuf, geom, R, case, seq, ["ties", "zero_residual", "c_midpoint"], 91)
    assert gpu.status.tolist() == [0, 0, 0, 0]
    print(f"ragged lengths: decode {worst:.2e}, fused {worst_f:.2e}; bytes equal")

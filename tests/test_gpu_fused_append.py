"""GPU: the anchor-loop call that also appends the current token
(rq_decode_attention_append).

Bars, step after step over consecutive slots (word and tile boundaries crossed):
  * against the same library's two separate calls -- rq_decode_attention for
    loop P-1, then rq_append with n_tokens = 1 -- the same output bits and the
    same cache bytes;
  * against the oracle's decode_attention_append: output max |gpu - oracle|
    <= 2e-3 and every cache byte equal (the oracle takes the residual in the
    device's float32 precision, as in the append parity tests).
"""
import math

import numpy as np
import pytest

import oracle
import synth
from rq_harness import Case, GpuCache, kv_for, rotation32

pytestmark = pytest.mark.gpu

ATOL = 2e-3


def _geom(case: Case):
    return oracle.Geometry(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax)


# d, g, loops per group, chained, scaling, rotation, batch, heads
CASES = [
    (128, 32, 4, False, "ls", "dense", 3, 2),
    (128, 16, 4, True, "ls", "dense", 2, 3),
    (96, 32, 4, False, "norm", "dense", 2, 2),
    (96, 16, 8, False, "ls", "dense", 2, 2),
    (128, 32, 16, False, "ls", "dense", 1, 2),
    (128, 32, 4, True, "norm", "dense", 2, 2),
    (128, 32, 8, False, "ls", "hadamard", 2, 2),
    (128, 32, 4, True, "ls", "hadamard", 2, 2),
]


@pytest.mark.parametrize("d,g,P,chained,scaling,rotation,B,H", CASES)
def test_fused_call_equals_decode_then_append_and_the_oracle(d, g, P, chained, scaling, rotation, B, H):
    case = Case(L=2, P=P, G=1, H=H, d=d, g=g, B=B, Nmax=192, chained=chained, scaling=scaling, seed=40 + P,
                rotation=rotation)
    R32, R = rotation32(d, kind=rotation)
    sep, fused = GpuCache(case, R32), GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    base = P == 4
    # rows of different lengths (121 and 130 tokens: mid-word and mid-tile slots next)
    start = np.array([0, 9, 0][:B], dtype=np.int64)
    n0 = 121
    kvb, kv = kv_for(case, 7, n0, base)
    for c in (sep, fused):
        c.append(1, 0, kvb, start)
    oracle.append(obuf, geom, R, 1, 0, kv, start, chained=chained, scaling=scaling, rotation=rotation)
    seq = start + n0
    scale = 1.0 / math.sqrt(d)
    worst = 0.0
    for step in range(8):
        kvb_c, kv_c = kv_for(case, 100 + step, 1, base)          # [P, 2, B, H, 1, d]
        qb, q = synth.queries(200 + step, B, H, d)
        out_s = sep.decode(1, 0, P - 1, qb, kvb_c[P - 1, 0, :, :, 0], kvb_c[P - 1, 1, :, :, 0], seq, scale)
        sep.append(1, 0, kvb_c, seq)
        out_f = fused.decode_append(1, 0, qb, kvb_c[..., 0, :], seq, scale)
        ref, ok = oracle.decode_attention_append(obuf, geom, R, 1, 0, q, kv_c[..., 0, :], seq, scale,
                                                 chained=chained, scaling=scaling, rotation=rotation)
        assert ok.all()
        o_s, o_f = out_s.cpu().numpy(), out_f.cpu().numpy()
        assert np.array_equal(o_s, o_f), f"step {step}: fused output differs from the two calls"
        err = float(np.abs(o_f - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"step {step}: max |gpu - oracle| = {err:.3e}"
        g_s, g_f = sep.bytes_host(), fused.bytes_host()
        assert np.array_equal(g_s, g_f), f"step {step}: {int((g_s != g_f).sum())} bytes differ from the two calls"
        assert np.array_equal(g_f, obuf), f"step {step}: {int((g_f != obuf).sum())} bytes differ from the oracle"
        seq = seq + 1
    assert sep.status.tolist() == [0, 0, 0, 0] and fused.status.tolist() == [0, 0, 0, 0]
    print(f"d={d} g={g} P={P} chained={chained} {scaling} {rotation}: worst max-abs error {worst:.3e}; "
          f"bytes equal")


def test_fused_call_empty_rows_and_capacity():
    """An empty row gets its first token at slot 0; a row with one free slot fills
    the last slot; a row at capacity is attended but not appended (status word
    [1] = 1, its bytes unchanged)."""
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=4, Nmax=128, seed=61)
    R32, R = rotation32(128)
    gpu = GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    kvb, kv = kv_for(case, 62, 100)
    start = np.array([0, 0, 28, 27], dtype=np.int64)     # row 2 fills the capacity, row 3 all but one slot
    gpu.append(0, 0, kvb, start)
    oracle.append(obuf, geom, R, 0, 0, kv, start)
    seq = np.array([0, 100, 128, 127])
    kvb_c, kv_c = kv_for(case, 63, 1)
    qb, q = synth.queries(64, 4, 2, 128)
    out = gpu.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, 0.09).cpu().numpy()
    ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, kv_c[..., 0, :], seq, 0.09)
    assert ok.tolist() == [True, True, False, True]
    assert np.abs(out - ref).max() <= ATOL
    assert np.array_equal(out[0], kv_c[3, 1, 0, :, 0].astype(np.float32))   # current token alone
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    st = gpu.status.cpu().numpy()
    assert st[0] == 0 and st[1] == 1


@pytest.mark.parametrize("chained", [False, True])
def test_fused_call_with_many_partials_per_head(chained):
    """Long rows at batch 1: every 128-token unit has its own decode CTA, so a
    (row, head) has 24 partial states, more than the merge combines in one
    batch.  The fused call still equals rq_decode_attention + rq_append bit for
    bit, and the oracle within 2e-3 (every cache byte equal)."""
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=1, Nmax=3200, chained=chained, seed=71)
    R32, R = rotation32(128)
    sep, fused = GpuCache(case, R32), GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    start = np.array([0], dtype=np.int64)
    n0 = 3050                                   # 24 units: 23 full, one of 106 tokens
    kvb, kv = kv_for(case, 72, n0)
    for c in (sep, fused):
        c.append(0, 0, kvb, start)
    oracle.append(obuf, geom, R, 0, 0, kv, start, chained=chained)
    seq = start + n0
    scale = 1.0 / math.sqrt(128)
    for step in range(2):
        kvb_c, kv_c = kv_for(case, 300 + step, 1)
        qb, q = synth.queries(400 + step, 1, 2, 128)
        out_s = sep.decode(0, 0, 3, qb, kvb_c[3, 0, :, :, 0], kvb_c[3, 1, :, :, 0], seq, scale)
        sep.append(0, 0, kvb_c, seq)
        out_f = fused.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, scale)
        ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, kv_c[..., 0, :], seq, scale,
                                                 chained=chained)
        assert ok.all()
        o_s, o_f = out_s.cpu().numpy(), out_f.cpu().numpy()
        assert np.array_equal(o_s, o_f), f"step {step}: fused output differs from the two calls"
        err = float(np.abs(o_f - ref).max())
        assert err <= ATOL, f"step {step}: max |gpu - oracle| = {err:.3e}"
        g_f = fused.bytes_host()
        assert np.array_equal(sep.bytes_host(), g_f)
        assert np.array_equal(g_f, obuf), f"step {step}: {int((g_f != obuf).sum())} bytes differ from the oracle"
        seq = seq + 1
    assert fused.status.tolist() == [0, 0, 0, 0]


def test_fused_call_with_more_coding_ctas_than_sms():
    """Batch 2 x 80 heads: 320 token-coding CTAs, more than the GPU's SMs, so the
    call runs the 64-register anchor-only decode kernel beside them.  Outputs and
    cache bytes equal the separate calls (the 72-register kernel, then
    rq_append) bit for bit, and the oracle within 2e-3."""
    import torch
    H = 80
    assert 2 * 2 * H > torch.cuda.get_device_properties(0).multi_processor_count
    case = Case(L=1, P=4, G=1, H=H, d=128, g=32, B=2, Nmax=256, seed=73)
    R32, R = rotation32(128)
    sep, fused = GpuCache(case, R32), GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    start = np.array([0, 17], dtype=np.int64)
    n0 = 150
    kvb, kv = kv_for(case, 74, n0)
    for c in (sep, fused):
        c.append(0, 0, kvb, start)
    oracle.append(obuf, geom, R, 0, 0, kv, start)
    seq = start + n0
    scale = 1.0 / math.sqrt(128)
    for step in range(2):
        kvb_c, kv_c = kv_for(case, 500 + step, 1)
        qb, q = synth.queries(600 + step, 2, H, 128)
        out_s = sep.decode(0, 0, 3, qb, kvb_c[3, 0, :, :, 0], kvb_c[3, 1, :, :, 0], seq, scale)
        sep.append(0, 0, kvb_c, seq)
        out_f = fused.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, scale)
        ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, kv_c[..., 0, :], seq, scale)
        assert ok.all()
        o_s, o_f = out_s.cpu().numpy(), out_f.cpu().numpy()
        assert np.array_equal(o_s, o_f), f"step {step}: fused output differs from the two calls"
        err = float(np.abs(o_f - ref).max())
        assert err <= ATOL, f"step {step}: max |gpu - oracle| = {err:.3e}"
        g_f = fused.bytes_host()
        assert np.array_equal(sep.bytes_host(), g_f)
        assert np.array_equal(g_f, obuf), f"step {step}: {int((g_f != obuf).sum())} bytes differ from the oracle"
        seq = seq + 1
    assert fused.status.tolist() == [0, 0, 0, 0]

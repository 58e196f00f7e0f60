"""GPU: the edges of the supported shapes.

  * a loop group of one loop (the anchor alone, no residual planes): appends,
    the attention call and the fused anchor-loop call, every byte and output
    against the oracle;
  * the largest batch one decode call takes (RQ_MAX_DECODE_BATCH rows, ragged
    lengths including empty rows), plain and fused calls against the oracle;
    one row more is refused with RQ_ERR_UNSUPPORTED before any launch;
  * an append whose batch x heads passes its grid limit is refused the same way.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from rq_harness import Case, GpuCache, kv_for, rotation32

pytestmark = pytest.mark.gpu

ATOL = 2e-3
MAX_BATCH = 256   # RQ_MAX_DECODE_BATCH in rq.h


def _geom(case: Case):
    return oracle.Geometry(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax)


def test_one_loop_group_is_the_anchor_alone():
    case = Case(L=1, P=1, G=1, H=2, d=128, g=32, B=2, Nmax=192, seed=95)
    R32, R = rotation32(case.d)
    gpu = GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    kvb, kv = kv_for(case, 96, 120, anchor_is_base=False)
    start = np.array([0, 7], dtype=np.int64)
    gpu.append(0, 0, kvb, start)
    oracle.append(obuf, geom, R, 0, 0, kv, start)
    seq = start + 120
    qb, q = synth.queries(97, 2, 2, 128)
    kvb_c, kv_c = kv_for(case, 98, 1, anchor_is_base=False)
    scale = 1 / math.sqrt(128)
    out = gpu.decode(0, 0, 0, qb, kvb_c[0, 0, :, :, 0], kvb_c[0, 1, :, :, 0], seq, scale).cpu().numpy()
    ref = oracle.decode_attention(obuf, geom, R, 0, 0, 0, q, kv_c[0, 0, :, :, 0], kv_c[0, 1, :, :, 0], seq, scale)
    assert np.abs(out - ref).max() <= ATOL
    out = gpu.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, scale).cpu().numpy()
    ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, kv_c[..., 0, :], seq, scale)
    assert ok.all() and np.abs(out - ref).max() <= ATOL
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    assert gpu.status.tolist() == [0, 0, 0, 0]


def test_largest_decode_batch():
    """RQ_MAX_DECODE_BATCH rows of one head; sampled rows checked against the
    oracle on a one-row cache of the same tokens (a row's region does not
    depend on the batch), bytes and outputs, for a plain and a fused call."""
    import decode_attention_rq_gb300 as rq
    case = Case(L=1, P=4, G=1, H=1, d=128, g=32, B=MAX_BATCH, Nmax=192, seed=99)
    R32, R = rotation32(case.d)
    gpu = GpuCache(case, R32)
    n = 70
    kvb, kv = kv_for(case, 100, n)                          # [P, 2, B, 1, n, d]
    gpu.append(0, 0, kvb, np.zeros(MAX_BATCH, dtype=np.int64))
    rng = np.random.default_rng(101)
    seq = rng.integers(0, n + 1, size=MAX_BATCH)
    rows = [0, 1, 2, 77, 200, MAX_BATCH - 1]
    seq[rows] = [0, n, 1, 64, 65, 33]
    scale = 1 / math.sqrt(128)
    qb1, q1 = synth.queries(102, MAX_BATCH, 1, 128)
    kvb_c, kv_c = kv_for(case, 104, 1)                      # [P, 2, B, 1, 1, d]
    out_res = gpu.decode(0, 0, 1, qb1, kvb_c[1, 0, :, :, 0], kvb_c[1, 1, :, :, 0], seq, scale).cpu().numpy()
    qb3, q3 = synth.queries(103, MAX_BATCH, 1, 128)
    out_fused = gpu.decode_append(0, 0, qb3, kvb_c[..., 0, :], seq, scale).cpu().numpy()
    gbuf = gpu.bytes_host()
    geom = oracle.Geometry(1, 4, 1, 1, 128, 32, MAX_BATCH, 192)
    one = oracle.Geometry(1, 4, 1, 1, 128, 32, 1, 192)
    for b in rows:
        obuf = np.zeros(one.total_bytes, dtype=np.uint8)
        oracle.append(obuf, one, R, 0, 0, kv[:, :, b:b + 1], [0])
        sl = seq[b:b + 1]
        ref = oracle.decode_attention(obuf, one, R, 0, 0, 1, q1[b:b + 1], kv_c[1, 0, b:b + 1, :, 0],
                                      kv_c[1, 1, b:b + 1, :, 0], sl, scale)
        assert np.abs(out_res[b] - ref[0]).max() <= ATOL, f"row {b}"
        ref, ok = oracle.decode_attention_append(obuf, one, R, 0, 0, q3[b:b + 1], kv_c[:, :, b:b + 1, :, 0], sl,
                                                 scale)
        assert ok.all() and np.abs(out_fused[b] - ref[0]).max() <= ATOL, f"row {b} (fused)"
        off = geom.region_offset(0, 0, b, 0)
        assert np.array_equal(gbuf[off:off + one.region], obuf), f"row {b}: cache bytes differ"
    assert gpu.status.tolist() == [0, 0, 0, 0]
    # one row more than a call may cover
    big = Case(L=1, P=4, G=1, H=1, d=128, g=32, B=MAX_BATCH + 8, Nmax=64, seed=1)
    gbig = GpuCache(big, R32)
    qb, _ = synth.queries(108, MAX_BATCH + 1, 1, 128)
    kvb_b, _ = kv_for(big, 109, 1)
    with pytest.raises(rq.RqError) as e:
        gbig.decode(0, 0, 0, qb, kvb_b[0, 0, :MAX_BATCH + 1, :, 0], kvb_b[0, 1, :MAX_BATCH + 1, :, 0],
                    np.zeros(MAX_BATCH + 1), scale, batch=MAX_BATCH + 1)
    assert e.value.status == 6   # RQ_ERR_UNSUPPORTED


def test_append_grid_limit_is_refused_before_any_launch():
    """rq_append puts (row, head) pairs on a grid dimension of at most 65535: a
    batch x heads above it returns RQ_ERR_UNSUPPORTED (nothing is launched, the
    cache stays zero); one pair fewer is accepted."""
    import torch
    import decode_attention_rq_gb300 as rq
    H, d, Nmax = 16, 128, 64
    B = 65536 // H                                  # 4096 rows x 16 heads = 65536 pairs
    case = Case(L=1, P=1, G=1, H=H, d=d, g=32, B=B, Nmax=Nmax, seed=3)
    R32, _ = rotation32(d)
    gpu = GpuCache(case, R32)
    kv = torch.zeros((1, 2, B, H, 1, d), dtype=torch.bfloat16, device="cuda:0")
    seq = torch.zeros(B, dtype=torch.int32, device="cuda:0")
    with pytest.raises(rq.RqError) as e:
        rq.rq_append(gpu.handle, 0, 0, B, kv, seq, 1, gpu.status)
    assert e.value.status == 6   # RQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert not gpu.buf.any()
    rq.rq_append(gpu.handle, 0, 0, B - 1, kv[:, :, :B - 1].contiguous(), seq, 1, gpu.status)   # 65520 pairs: accepted
    torch.cuda.synchronize()
    assert gpu.status.tolist() == [0, 0, 0, 0]

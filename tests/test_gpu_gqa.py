"""GPU: grouped-query attention (rq_config.num_query_heads a multiple of num_heads).

Query head qh attends with KV head qh / (Hq / H).  Bars:
  * every loop's output within 2e-3 of the oracle's grouped-query attention;
  * bit for bit the output of the same calls on a multi-head cache whose heads
    are copies of the KV heads (head qh = KV head qh / (Hq / H));
  * the anchor-loop call's token append (one append per KV head) leaves every
    cache byte equal to the oracle's.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from rq_harness import Case, GpuCache, kv_for, rotation32

pytestmark = pytest.mark.gpu

ATOL = 2e-3


# Hq / H = 2 and 4 run the multi-query kernel with two and four heads per work
# unit, 8 with four heads in two groups; the chained case's loops 0 and 1 (three
# and two residual planes) take the per-head kernel, its loops 2 and 3 the
# multi-query one.
@pytest.mark.parametrize("d,g,H,Hq,chained", [(128, 32, 2, 4, False), (128, 32, 2, 8, False), (96, 16, 3, 6, True),
                                              (128, 16, 1, 8, False), (96, 32, 2, 8, False), (128, 32, 3, 6, True)])
def test_grouped_query_attention(d, g, H, Hq, chained):
    case = Case(L=1, P=4, G=1, H=H, d=d, g=g, B=2, Nmax=256, seed=90, chained=chained, Hq=Hq)
    mha = Case(L=1, P=4, G=1, H=Hq, d=d, g=g, B=2, Nmax=256, seed=90, chained=chained)
    qpk = Hq // H
    R32, R = rotation32(d)
    gqa_dev, mha_dev = GpuCache(case, R32), GpuCache(mha, R32)
    geom = oracle.Geometry(1, 4, 1, H, d, g, 2, 256)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    kvb, kv = kv_for(case, 91, 150)                          # [P, 2, B, H, n, d]
    start = np.array([0, 40], dtype=np.int64)
    gqa_dev.append(0, 0, kvb, start)
    mha_dev.append(0, 0, torch.repeat_interleave(kvb, qpk, dim=3), start)
    oracle.append(obuf, geom, R, 0, 0, kv, start, chained=chained)
    seq = start + 150
    scale = 1.0 / math.sqrt(d)
    worst = 0.0
    for loop in range(4):
        qb, q = synth.queries(92 + loop, 2, Hq, d)
        kvb_c, kv_c = kv_for(case, 93 + loop, 1)             # [P, 2, B, H, 1, d]
        if loop < 3:
            kcb, vcb = kvb_c[loop, 0, :, :, 0], kvb_c[loop, 1, :, :, 0]
            out = gqa_dev.decode(0, 0, loop, qb, kcb, vcb, seq, scale).cpu().numpy()
            out_m = mha_dev.decode(0, 0, loop, qb, torch.repeat_interleave(kcb, qpk, dim=1),
                                   torch.repeat_interleave(vcb, qpk, dim=1), seq, scale).cpu().numpy()
            ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kv_c[loop, 0, :, :, 0],
                                          kv_c[loop, 1, :, :, 0], seq, scale, chained=chained)
        else:   # the anchor loop's call also appends the token (per KV head)
            out = gqa_dev.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, scale).cpu().numpy()
            out_m = mha_dev.decode_append(0, 0, qb, torch.repeat_interleave(kvb_c[..., 0, :], qpk, dim=3), seq,
                                          scale).cpu().numpy()
            ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, kv_c[..., 0, :], seq, scale,
                                                     chained=chained)
            assert ok.all()
        assert out.shape == (2, Hq, d)
        assert np.array_equal(out, out_m), f"loop {loop}: differs from multi-head over copied heads"
        err = float(np.abs(out - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"loop {loop}: max |gpu - oracle| = {err:.3e}"
    gbuf = gqa_dev.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    assert gqa_dev.status.tolist() == [0, 0, 0, 0]
    print(f"GQA H={H} Hq={Hq} d={d} chained={chained}: worst max-abs error {worst:.3e}; cache bytes equal")


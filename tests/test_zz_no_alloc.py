"""rq_decode_attention_noalloc against rq_decode_attention (GPU).

The no-alloc entry point serves callers that cannot allocate device memory --
a plugin whose host application owns every device buffer, or a process whose
memory budget is fixed before decoding starts.  It must give what the
workspace-taking entry point gives, on consecutive calls (the built-in array
keeps the previous call's contents, so each call has to clear what must
start at zero), and must refuse a batch its fixed array cannot hold.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run on its own.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from rq_harness import Case, GpuCache, kv_for, rotation32

pytestmark = pytest.mark.gpu

ATOL = 2e-3   # against the oracle: the decode parity tests' bar


def _inputs(case, seed):
    gen = torch.Generator().manual_seed(seed)
    shape = (case.B, case.H, case.d)
    q, kc, vc = (torch.randn(shape, generator=gen).to(torch.bfloat16).cuda() for _ in range(3))
    return q, kc, vc


def test_noalloc_matches_workspace_call_twice_in_a_row():
    import decode_attention_rq_gb300 as rq
    case = Case(L=1, P=4, G=1, H=4, d=128, g=32, B=3, Nmax=768, seed=11)
    R32, R = rotation32(case.d)
    gpu = GpuCache(case, R32)
    kvb, kv = kv_for(case, seed=case.seed, ntok=700)
    gpu.append(0, 0, kvb, [0] * case.B)
    geom = oracle.Geometry(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    oracle.append(obuf, geom, R, 0, 0, kv, np.zeros(case.B, dtype=np.int64))
    lens = [700, 129, 0]                       # several tiles, a ragged tail, an empty row
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q, kc, vc = _inputs(case, 5)
    scale = 1 / math.sqrt(case.d)
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    for loop in (1, 3):                        # a residual loop and the anchor loop
        ref = gpu.decode(0, 0, loop, q, kc, vc, lens, scale)
        exact = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q.double().cpu().numpy(),
                                        kc.double().cpu().numpy(), vc.double().cpu().numpy(), lens, scale)
        for call in range(2):
            out = torch.full((case.B, case.H, case.d), float("nan"), device="cuda")
            rq.rq_decode_attention_noalloc(gpu.handle, 0, 0, loop, case.B, q, kc, vc, sl, scale, out,
                                           status)
            torch.cuda.synchronize()
            # the same kernels on the same inputs: the same bits as the workspace call
            assert torch.equal(out, ref), (loop, call, (out - ref).abs().max().item())
            err = float(np.abs(out.cpu().numpy() - exact).max())
            assert err <= ATOL, (loop, call, err)
            assert status.tolist() == [0, 0, 0, 0], (loop, call, status.tolist())
    gpu.close()


def test_noalloc_refuses_a_batch_beyond_its_array():
    import decode_attention_rq_gb300 as rq
    case = Case(L=1, P=4, G=1, H=16, d=128, g=32, B=128, Nmax=64, seed=3)
    R32, _ = rotation32(case.d)
    gpu = GpuCache(case, R32)
    assert rq.rq_decode_workspace_bytes(gpu.cfg, case.B) > rq.RQ_NOALLOC_WORKSPACE_BYTES
    q, kc, vc = _inputs(case, 6)
    sl = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    out = torch.empty((case.B, case.H, case.d), dtype=torch.float32, device="cuda")
    with pytest.raises(rq.RqError) as e:
        rq.rq_decode_attention_noalloc(gpu.handle, 0, 0, 0, case.B, q, kc, vc, sl, 0.1, out)
    assert e.value.status == 4                 # RQ_ERR_WORKSPACE
    # a batch that fits still runs (all rows empty: the output is the current V)
    b = 8
    rq.rq_decode_attention_noalloc(gpu.handle, 0, 0, 0, b, q, kc, vc, sl, 0.1, out)
    torch.cuda.synchronize()
    assert torch.equal(out[:b], vc[:b].float())
    gpu.close()

"""Parity at the full workload sizes, in the launch configuration the benchmark times (GPU).

For each workload (Ouro-shaped 8k batch 4, 16k batch 2 and 4, Huginn-shaped,
two batch-sweep points, one of them chained), the device cache of one layer is
filled at the workload's batch, head count and context; a few (row, head)
slices are drawn from synth.looped_kv_slice and the rest from the device
generator.  The decode calls run at the full batch (so the grid, the work
split and the merge are those of the benchmark), with one row shorter than the
others; as in the benchmark's step, the anchor loop's call also appends the
current token (rq_decode_attention_append).  For every sampled slice the
oracle compresses the same values on its own, attends over them for every
loop and appends the token; the test checks

  * the slice's cache region, byte for byte (codes, metadata, coefficients,
    the appended slot included);
  * the decode output of every loop, max |gpu - oracle| <= 2e-3.

The oracle slices run in a spawned process pool while the device side runs.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from fullsize_oracle import slice_job

pytestmark = pytest.mark.gpu

ATOL = 2e-3
CHUNK = 2048          # tokens per device append while filling the cache
SHORT = 37            # the last row holds this many tokens fewer


def _cases():
    W = synth.WORKLOADS
    # name -> (workload, chained, samples [(layer, group, row, head)], seed)
    return {
        "ouro8k": (W["ouro8k"], False, [(0, 0, 0, 5), (0, 0, 3, 11)], 101),
        "ouro16k_b2": (W["ouro16k_b2"], False, [(0, 0, 1, 7)], 102),
        "ouro16k_b4": (W["ouro16k_b4"], False, [(0, 0, 2, 15)], 103),
        "huginn": (W["huginn"], False, [(0, 0, 0, 3), (0, 7, 1, 54)], 104),
        "sweep_b128_g32": (synth.sweep_workload(128, 32), False, [(0, 0, 127, 9)], 105),
        "sweep_b32_g16_chained": (synth.sweep_workload(32, 16), True, [(0, 0, 31, 2)], 106),
    }


def _gqa_cases():
    """Grouped-query heads at the Ouro 8k batch-4 size: Hq query heads over the
    16 KV heads (the multi-query kernel, 2 or 4 query heads per unit); samples
    (layer, group, row, KV head, query head) with the query head on that KV head."""
    W = synth.WORKLOADS
    return {
        "ouro8k_hq32": (W["ouro8k"], 32, [(0, 0, 1, 5, 11), (0, 0, 3, 12, 24)], 107),
        "ouro8k_hq64": (W["ouro8k"], 64, [(0, 0, 0, 9, 39), (0, 0, 2, 15, 60)], 108),
    }


def _q_inputs(w, Hq, seed):
    """Per loop: queries [B, Hq, d] (bf16, float64) and the current token's K/V per KV head."""
    B, H, d = w.batch, w.num_heads, w.head_dim
    return [(synth.queries(seed * 10 + loop, B, Hq, d), synth.queries(seed * 10 + 1000 + loop, B, H, d),
             synth.queries(seed * 10 + 2000 + loop, B, H, d)) for loop in range(w.loops_per_group)]


def _inputs(w, seed):
    """Per loop: queries and the current token's K/V for every (row, head): bf16 and float64."""
    B, H, d = w.batch, w.num_heads, w.head_dim
    out = []
    for loop in range(w.loops_per_group):
        out.append(tuple(synth.queries(seed * 10 + 1000 * k + loop, B, H, d) for k in range(3)))
    return out


def _seq_lens(w):
    s = np.full(w.batch, w.context, dtype=np.int64)
    s[-1] = w.context - SHORT
    return s


@pytest.fixture(scope="module")
def oracle_results():
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(processes=max(1, min(8, os.cpu_count() or 1)))
    res = {}
    for name, (w, chained, samples, seed) in _cases().items():
        ins = _inputs(w, seed)
        seq = _seq_lens(w)
        for (layer, group, b, h) in samples:
            q = np.stack([ins[l][0][1][b, h] for l in range(w.loops_per_group)])
            kc = np.stack([ins[l][1][1][b, h] for l in range(w.loops_per_group)])
            vc = np.stack([ins[l][2][1][b, h] for l in range(w.loops_per_group)])
            args = (w, seed, layer, group, b, h, w.context, w.context + 64, int(seq[b]), chained, q, kc, vc,
                    synth.softmax_scale(w.head_dim))
            res[(name, layer, group, b, h)] = pool.apply_async(slice_job, (args,))
    for name, (w, Hq, samples, seed) in _gqa_cases().items():
        ins = _q_inputs(w, Hq, seed)
        seq = _seq_lens(w)
        for (layer, group, b, h, qh) in samples:
            q = np.stack([ins[l][0][1][b, qh] for l in range(w.loops_per_group)])
            kc = np.stack([ins[l][1][1][b, h] for l in range(w.loops_per_group)])
            vc = np.stack([ins[l][2][1][b, h] for l in range(w.loops_per_group)])
            args = (w, seed, layer, group, b, h, w.context, w.context + 64, int(seq[b]), False, q, kc, vc,
                    synth.softmax_scale(w.head_dim))
            res[(name, layer, group, b, h, qh)] = pool.apply_async(slice_job, (args,))
    pool.close()
    yield res
    pool.terminate()
    pool.join()


def _device_case(w, chained, samples, seed):
    import decode_attention_rq_gb300 as rq
    dev = "cuda:0"
    P, H, d, g, B, N = w.loops_per_group, w.num_heads, w.head_dim, w.group_size, w.batch, w.context
    groups = sorted({s[1] for s in samples})
    G = max(groups) + 1
    cap = N + 64
    cfg = rq.rq_config(1, P, G, H, d, g, B, cap, rq.RQ_MODE_CHAINED if chained else rq.RQ_MODE_SHARED)
    nbytes = rq.rq_cache_bytes(cfg)
    buf = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    R = torch.from_numpy(synth.rotation(d).astype(np.float32)).to(dev)
    handle = rq.rq_cache_create(cfg, buf, nbytes, R)
    ws_bytes = rq.rq_decode_workspace_bytes(cfg, B)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    status = ws[:16].view(torch.int32)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    slices = {s: synth.looped_kv_slice(seed, w, N, *s)[0].to(dev) for s in samples}
    for grp in groups:
        for c0 in range(0, N, CHUNK):
            n = min(CHUNK, N - c0)
            kv = synth.looped_kv_torch(gen, w, B, n, dev)
            for (layer, gg, b, h), t in slices.items():
                if gg == grp:
                    kv[:, :, b, h] = t[:, :, c0:c0 + n]
            seq = torch.full((B,), c0, dtype=torch.int32, device=dev)
            rq.rq_append(handle, 0, grp, B, kv, seq, n, status)
            del kv
    torch.cuda.synchronize()
    assert int(status[1]) == 0, "append reported a capacity overflow"
    sl = torch.as_tensor(_seq_lens(w).astype(np.int32), device=dev)
    scale = synth.softmax_scale(d)
    ins = _inputs(w, seed)
    outs = {}
    # the current token of every loop, [P, 2, B, H, d]: the anchor-loop call appends it
    kv_all = torch.stack([torch.stack([ins[l][1][0], ins[l][2][0]]) for l in range(P)]).to(dev).contiguous()
    for loop in range(P):
        (q, _), (kc, _), (vc, _) = ins[loop]
        q, kc, vc = q.to(dev), kc.to(dev), vc.to(dev)
        for grp in groups:
            out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
            if loop < P - 1:
                rq.rq_decode_attention(handle, 0, grp, loop, B, q, kc, vc, sl, scale, out, ws, ws_bytes)
            else:
                rq.rq_decode_attention_append(handle, 0, grp, B, q, kv_all, sl, scale, out, ws, ws_bytes)
            outs[(grp, loop)] = out.cpu().numpy()
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0, 0, 0]
    geom = oracle.Geometry(1, P, G, H, d, g, B, cap)
    regions = {}
    for s in samples:
        off = geom.region_offset(*s)
        regions[s] = buf[off: off + geom.region].cpu().numpy()
    rq.rq_cache_destroy(handle)
    del buf, ws
    torch.cuda.empty_cache()
    return regions, outs


@pytest.mark.parametrize("name", list(_cases()))
def test_fullsize_sampled_parity(name, oracle_results):
    w, chained, samples, seed = _cases()[name]
    regions, outs = _device_case(w, chained, samples, seed)
    worst = 0.0
    for s in samples:
        layer, group, b, h = s
        obuf, oout = oracle_results[(name,) + s].get(timeout=1800)
        diff = int((regions[s] != obuf).sum())
        assert diff == 0, f"{name} {s}: {diff} of {obuf.size} cache bytes differ"
        for loop in range(w.loops_per_group):
            err = float(np.abs(outs[(group, loop)][b, h] - oout[loop]).max())
            worst = max(worst, err)
            assert err <= ATOL, f"{name} {s} loop {loop}: max |gpu - oracle| = {err:.3e}"
    print(f"{name}: worst max-abs error {worst:.3e} over {len(samples)} slices x {w.loops_per_group} loops; "
          f"cache bytes equal")


def _gqa_device_case(w, Hq, samples, seed):
    import decode_attention_rq_gb300 as rq
    dev = "cuda:0"
    P, H, d, g, B, N = w.loops_per_group, w.num_heads, w.head_dim, w.group_size, w.batch, w.context
    cap = N + 64
    cfg = rq.rq_config(1, P, 1, H, d, g, B, cap, rq.RQ_MODE_SHARED, Hq)
    nbytes = rq.rq_cache_bytes(cfg)
    buf = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    R = torch.from_numpy(synth.rotation(d).astype(np.float32)).to(dev)
    handle = rq.rq_cache_create(cfg, buf, nbytes, R)
    ws_bytes = rq.rq_decode_workspace_bytes(cfg, B)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    status = ws[:16].view(torch.int32)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    slices = {s[:4]: synth.looped_kv_slice(seed, w, N, *s[:4])[0].to(dev) for s in samples}
    for c0 in range(0, N, CHUNK):
        n = min(CHUNK, N - c0)
        kv = synth.looped_kv_torch(gen, w, B, n, dev)
        for (layer, gg, b, h), t in slices.items():
            kv[:, :, b, h] = t[:, :, c0:c0 + n]
        seq = torch.full((B,), c0, dtype=torch.int32, device=dev)
        rq.rq_append(handle, 0, 0, B, kv, seq, n, status)
        del kv
    torch.cuda.synchronize()
    sl = torch.as_tensor(_seq_lens(w).astype(np.int32), device=dev)
    scale = synth.softmax_scale(d)
    ins = _q_inputs(w, Hq, seed)
    kv_all = torch.stack([torch.stack([ins[l][1][0], ins[l][2][0]]) for l in range(P)]).to(dev).contiguous()
    outs = {}
    for loop in range(P):
        (q, _), (kc, _), (vc, _) = ins[loop]
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
        if loop < P - 1:
            rq.rq_decode_attention(handle, 0, 0, loop, B, q.to(dev), kc.to(dev), vc.to(dev), sl, scale, out, ws,
                                   ws_bytes)
        else:
            rq.rq_decode_attention_append(handle, 0, 0, B, q.to(dev), kv_all, sl, scale, out, ws, ws_bytes)
        outs[loop] = out.cpu().numpy()
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0, 0, 0]
    geom = oracle.Geometry(1, P, 1, H, d, g, B, cap)
    regions = {}
    for s in samples:
        off = geom.region_offset(*s[:4])
        regions[s] = buf[off: off + geom.region].cpu().numpy()
    rq.rq_cache_destroy(handle)
    del buf, ws
    torch.cuda.empty_cache()
    return regions, outs


@pytest.mark.parametrize("name", list(_gqa_cases()))
def test_fullsize_grouped_query_sampled_parity(name, oracle_results):
    """The multi-query kernel at the benchmark's size (every CTA takes several
    units and crosses head-group boundaries): sampled (row, query head) outputs
    of every loop within 2e-3 of the oracle, the KV head's region byte-equal
    (the appended slot included)."""
    w, Hq, samples, seed = _gqa_cases()[name]
    regions, outs = _gqa_device_case(w, Hq, samples, seed)
    worst = 0.0
    for s in samples:
        layer, group, b, h, qh = s
        obuf, oout = oracle_results[(name,) + s].get(timeout=1800)
        diff = int((regions[s] != obuf).sum())
        assert diff == 0, f"{name} {s}: {diff} of {obuf.size} cache bytes differ"
        for loop in range(w.loops_per_group):
            err = float(np.abs(outs[loop][b, qh] - oout[loop]).max())
            worst = max(worst, err)
            assert err <= ATOL, f"{name} {s} loop {loop}: max |gpu - oracle| = {err:.3e}"
    print(f"{name}: worst max-abs error {worst:.3e} over {len(samples)} slices x {w.loops_per_group} loops")

"""GPU: the paged (block-table) cache layout (rq_cache_create_paged).

The same tokens go into a paged cache (pages assigned by a shuffled table,
spare pages left unused, a table wider than needed with unused entries out of
range) and into the oracle's contiguous cache.  Bars:
  * the page pool equals oracle.paged_pool of the oracle's bytes, byte for byte,
    after prefill appends, a one-token append and the fused anchor-loop call;
  * every loop's attention output equals, bit for bit, the same call on a
    contiguous device cache holding the same tokens, and is within 2e-3 of the
    oracle's;
  * a table entry outside the pool for a tile in use is not followed: status
    word [2] is set, the call completes, the pool outside the pages in use is
    untouched.
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


class PagedCache(GpuCache):
    """GpuCache whose storage is a page pool addressed through a block table."""

    def __init__(self, case: Case, R32, table: np.ndarray, num_pages: int, device="cuda:0"):
        import decode_attention_rq_gb300 as rq
        self.rq, self.case, self.device = rq, case, device
        self.cfg = rq.rq_config(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax,
                                (rq.RQ_MODE_CHAINED if case.chained else rq.RQ_MODE_SHARED)
                                | (rq.RQ_MODE_HADAMARD if case.rotation == "hadamard" else 0), case.Hq)
        self.nbytes = rq.rq_cache_paged_bytes(self.cfg, num_pages)
        assert self.nbytes > 0
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)
        self.table = torch.as_tensor(np.ascontiguousarray(table, dtype=np.int32), device=device)
        self.R = None if case.rotation == "hadamard" else torch.from_numpy(R32).to(device)
        self.handle = rq.rq_cache_create_paged(self.cfg, num_pages, self.buf, self.nbytes, self.table,
                                               table.shape[1], self.R)
        self.ws_bytes = rq.rq_decode_workspace_bytes(self.cfg, case.B)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.status = self.ws[:16].view(torch.int32)


def _table(case: Case, extra_pages=5, extra_cols=2, seed=0):
    ntiles = -(-case.Nmax // 64)
    num_pages = case.B * ntiles + extra_pages
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)
    table = np.full((case.B, ntiles + extra_cols), num_pages + 1000, dtype=np.int64)   # unused: out of range
    table[:, :ntiles] = perm[: case.B * ntiles].reshape(case.B, ntiles)
    return table, num_pages


def _geom(case: Case):
    return oracle.Geometry(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax)


@pytest.mark.parametrize("chained,rotation", [(False, "dense"), (True, "dense"), (False, "hadamard")])
def test_paged_layout_matches_the_oracle_and_the_contiguous_cache(chained, rotation):
    case = Case(L=2, P=4, G=2, H=3, d=128, g=32, B=3, Nmax=256, seed=70, chained=chained, rotation=rotation)
    R32, R = rotation32(case.d, kind=rotation)
    table, num_pages = _table(case)
    paged, contig = PagedCache(case, R32, table, num_pages), GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    start = np.array([0, 5, 60], dtype=np.int64)
    n0 = 130
    for layer in range(case.L):
        for group in range(case.G):
            kvb, kv = kv_for(case, 700 + 10 * layer + group, n0)
            paged.append(layer, group, kvb, start)
            contig.append(layer, group, kvb, start)
            oracle.append(obuf, geom, R, layer, group, kv, start, chained=chained, rotation=rotation)
    pool = paged.bytes_host()
    want = oracle.paged_pool(obuf, geom, table, num_pages)
    assert np.array_equal(pool, want), f"{int((pool != want).sum())} pool bytes differ after the prefill"
    seq = start + n0
    scale = 1.0 / math.sqrt(case.d)
    worst = 0.0
    for layer, group in [(0, 1), (1, 0)]:
        for loop in range(case.P):
            qb, q = synth.queries(800 + loop, case.B, case.H, case.d)
            kvb_c, kv_c = kv_for(case, 900 + loop, 1)
            kcb, vcb = kvb_c[loop, 0, :, :, 0], kvb_c[loop, 1, :, :, 0]
            if loop < case.P - 1:
                out_p = paged.decode(layer, group, loop, qb, kcb, vcb, seq, scale).cpu().numpy()
                out_c = contig.decode(layer, group, loop, qb, kcb, vcb, seq, scale).cpu().numpy()
                ref = oracle.decode_attention(obuf, geom, R, layer, group, loop, q, kv_c[loop, 0, :, :, 0],
                                              kv_c[loop, 1, :, :, 0], seq, scale, chained=chained)
            else:   # the anchor loop's call also appends the token
                out_p = paged.decode_append(layer, group, qb, kvb_c[..., 0, :], seq, scale).cpu().numpy()
                out_c = contig.decode_append(layer, group, qb, kvb_c[..., 0, :], seq, scale).cpu().numpy()
                ref, ok = oracle.decode_attention_append(obuf, geom, R, layer, group, q, kv_c[..., 0, :], seq, scale,
                                                         chained=chained, rotation=rotation)
                assert ok.all()
            assert np.array_equal(out_p, out_c), f"layer {layer} loop {loop}: paged output differs"
            err = float(np.abs(out_p - ref).max())
            worst = max(worst, err)
            assert err <= ATOL, f"layer {layer} loop {loop}: max |gpu - oracle| = {err:.3e}"
    pool = paged.bytes_host()
    want = oracle.paged_pool(obuf, geom, table, num_pages)
    assert np.array_equal(pool, want), f"{int((pool != want).sum())} pool bytes differ after the fused calls"
    assert paged.status.tolist() == [0, 0, 0, 0] and contig.status.tolist() == [0, 0, 0, 0]
    print(f"paged chained={chained} {rotation}: worst max-abs error {worst:.3e}; pool bytes equal")


def test_paged_out_of_range_entry_is_not_followed():
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=2, Nmax=192, seed=71)
    R32, R = rotation32(case.d)
    table, num_pages = _table(case, extra_pages=0, extra_cols=0, seed=3)
    kvb, kv = kv_for(case, 710, 100)
    good = PagedCache(case, R32, table.copy(), num_pages)
    good.append(0, 0, kvb, [0, 0])
    bad_table = table.copy()
    bad_table[1, 1] = num_pages + 7          # row 1, tokens 64..127: in use
    bad = PagedCache(case, R32, bad_table, num_pages)
    bad.append(0, 0, kvb, [0, 0])
    torch.cuda.synchronize()
    assert int(bad.status[2]) == 1
    pool_bad, pool_good = bad.bytes_host(), good.bytes_host()
    # everything but the page row 1 tile 1 would have used is identical
    geom_pb = oracle.Geometry(1, 4, 1, 2, 128, 32, 2, 192)
    page_bytes = 2 * (2 * geom_pb.a_tile + 6 * geom_pb.r_tile)
    skip = int(table[1, 1])
    mask = np.ones(pool_good.size, bool)
    mask[skip * page_bytes + page_bytes // 2: (skip + 1) * page_bytes] = False   # head 1 of that page
    mask[skip * page_bytes: skip * page_bytes + page_bytes // 2] = False         # head 0 of that page
    assert np.array_equal(pool_bad[mask], pool_good[mask])
    assert not pool_bad[~mask].any()
    # decode over the bad tile reads page 0 instead, completes and flags it
    bad.status.zero_()
    qb, q = synth.queries(711, 2, 2, 128)
    out = bad.decode(0, 0, 1, qb, kvb[1, 0, :, :, 0], kvb[1, 1, :, :, 0], [100, 100], 0.09)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert int(bad.status[2]) == 1 and int(bad.status[0]) == 0


def test_paged_grouped_query_chained_eight_loops_hadamard():
    """The options together: paged layout, grouped-query heads (Hq = 2H), chained
    groups of 8 loops (a call reads up to seven residual planes), Walsh-Hadamard
    rotation.  Pool bytes equal the oracle's paged view after the prefill and
    after a fused anchor-loop call; every loop within 2e-3 of the oracle."""
    case = Case(L=1, P=8, G=1, H=2, d=128, g=32, B=2, Nmax=192, seed=73, chained=True, rotation="hadamard", Hq=4)
    R32, R = rotation32(case.d, kind="hadamard")
    table, num_pages = _table(case, seed=6)
    paged = PagedCache(case, R32, table, num_pages)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    start = np.array([0, 20], dtype=np.int64)
    kvb, kv = kv_for(case, 730, 100, anchor_is_base=False)
    paged.append(0, 0, kvb, start)
    oracle.append(obuf, geom, R, 0, 0, kv, start, chained=True, rotation="hadamard")
    assert np.array_equal(paged.bytes_host(), oracle.paged_pool(obuf, geom, table, num_pages))
    seq = start + 100
    scale = 1.0 / math.sqrt(case.d)
    worst = 0.0
    for loop in (0, 4, 7):
        qb, q = synth.queries(740 + loop, case.B, 4, case.d)
        kvb_c, kv_c = kv_for(case, 750 + loop, 1, anchor_is_base=False)
        if loop < 7:
            out = paged.decode(0, 0, loop, qb, kvb_c[loop, 0, :, :, 0], kvb_c[loop, 1, :, :, 0], seq, scale)
            ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kv_c[loop, 0, :, :, 0],
                                          kv_c[loop, 1, :, :, 0], seq, scale, chained=True)
        else:
            out = paged.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, scale)
            ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, kv_c[..., 0, :], seq, scale,
                                                     chained=True, rotation="hadamard")
            assert ok.all()
        err = float(np.abs(out.cpu().numpy() - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"loop {loop}: max |gpu - oracle| = {err:.3e}"
    assert np.array_equal(paged.bytes_host(), oracle.paged_pool(obuf, geom, table, num_pages))
    assert paged.status.tolist() == [0, 0, 0, 0]
    print(f"paged + GQA + chained P=8 + Hadamard: worst max-abs error {worst:.3e}; pool bytes equal")


@pytest.mark.parametrize("d,g,H,Hq", [(128, 32, 2, 4), (128, 16, 2, 8), (96, 32, 1, 4)])
def test_paged_grouped_query_multi_query_kernel(d, g, H, Hq):
    """Grouped-query heads on a paged cache, shared anchors: every call reads at
    most one residual plane, so all four loops run the multi-query kernel (2 or
    4 query heads per unit; Hq / H = 8 as two head groups).  Outputs bit-equal to
    the same calls on a contiguous cache and within 2e-3 of the oracle; the pool
    equals the oracle's paged view after the fused anchor-loop call."""
    case = Case(L=1, P=4, G=1, H=H, d=d, g=g, B=3, Nmax=320, seed=76, Hq=Hq)
    R32, R = rotation32(case.d)
    table, num_pages = _table(case, seed=9)
    paged, contig = PagedCache(case, R32, table, num_pages), GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    start = np.array([0, 33, 70], dtype=np.int64)
    kvb, kv = kv_for(case, 760, 200)
    paged.append(0, 0, kvb, start)
    contig.append(0, 0, kvb, start)
    oracle.append(obuf, geom, R, 0, 0, kv, start)
    seq = start + 200
    scale = 1.0 / math.sqrt(case.d)
    worst = 0.0
    for loop in range(4):
        qb, q = synth.queries(770 + loop, case.B, Hq, case.d)
        kvb_c, kv_c = kv_for(case, 780 + loop, 1)
        if loop < 3:
            kc, vc = kvb_c[loop, 0, :, :, 0], kvb_c[loop, 1, :, :, 0]
            out = paged.decode(0, 0, loop, qb, kc, vc, seq, scale).cpu().numpy()
            out_c = contig.decode(0, 0, loop, qb, kc, vc, seq, scale).cpu().numpy()
            ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kv_c[loop, 0, :, :, 0],
                                          kv_c[loop, 1, :, :, 0], seq, scale)
        else:
            out = paged.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, scale).cpu().numpy()
            out_c = contig.decode_append(0, 0, qb, kvb_c[..., 0, :], seq, scale).cpu().numpy()
            ref, ok = oracle.decode_attention_append(obuf, geom, R, 0, 0, q, kv_c[..., 0, :], seq, scale)
            assert ok.all()
        assert np.array_equal(out, out_c), f"loop {loop}: paged differs from contiguous"
        err = float(np.abs(out - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"loop {loop}: max |gpu - oracle| = {err:.3e}"
    assert np.array_equal(paged.bytes_host(), oracle.paged_pool(obuf, geom, table, num_pages))
    assert paged.status.tolist() == [0, 0, 0, 0]
    print(f"paged GQA d={d} g={g} Hq/H={Hq // H}: worst max-abs error {worst:.3e}")

"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Bars (the precision targets for this method and the oracle's readings):
  * every cache byte (INT4 and INT2 codes, E4M3 metadata, BF16 coefficients)
    equal to the oracle's.  The oracle takes the rotated residual in the
    device's reading (binary32: e rounded once, u_i an FMA chain in channel
    order), so the bytes must match exactly;
  * against the oracle's float64 reading of the same residual (no binary32
    rounding), test_residual_codes_against_the_float64_reading applies the
    boundary rule: anchor bytes and coefficients equal; a residual code or
    metadata byte may differ only where the float64 value lies at a rounding
    boundary (within 1e-3 of a code midpoint, 1e-4 relative of an E4M3
    midpoint), the code by one step, and rarely;
  * attention outputs: max |gpu - oracle| <= 2e-3 (float32 output, O(1) data).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import formats as F
from rq_harness import Case, GpuCache, kv_for, plane_views, rotation32

pytestmark = pytest.mark.gpu

ATOL = 2e-3


def _geom(case: Case):
    return oracle.Geometry(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax)


def _near_e4m3_midpoint(x, rel=1e-4):
    """True where x is within rel of an E4M3 rounding boundary (midpoint of two neighbours)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    codes, vals = oracle.formats.e4m3_all_finite()
    mids = (vals[:-1] + vals[1:]) / 2
    i = np.searchsorted(mids, x)
    d = np.full(x.shape, np.inf)
    for k in (i - 1, i):
        k = np.clip(k, 0, len(mids) - 1)
        d = np.minimum(d, np.abs(x - mids[k]))
    return d <= rel * np.maximum(x, 2.0 ** -9)


def check_residual_parity(gbuf, obuf, geom, comp_u, layer, group, n, B, H, chained=False, max_rate=1e-3):
    """comp_u[j]: oracle float64 rotated residual [2, B, H, n, d] for loop j."""
    g, d, ng = geom.group_size, geom.head_dim, geom.ng
    total, bad_codes, bad_groups, c_diff = 0, 0, 0, 0
    for b in range(B):
        for h in range(H):
            for kv in range(2):
                for j in range(geom.loops_per_group - 1):
                    gc, gs, go, gcb = oracle.read_plane_tokens(gbuf, geom, layer, group, b, h, kv, "res", j, n)
                    oc, os_, oo, ocb = oracle.read_plane_tokens(obuf, geom, layer, group, b, h, kv, "res", j, n)
                    total += gc.size
                    cd = gcb != ocb
                    c_diff += int(cd.sum())
                    if not chained:
                        assert not cd.any(), f"BF16 coefficient differs (b={b} h={h} kv={kv} j={j})"
                    u = comp_u[j][kv, b, h]                      # [n, d]
                    ug = u.reshape(n, ng, g)
                    meta_diff = (gs != os_) | (go != oo)         # [n, ng]
                    tok_c = cd[:, None] & np.ones((1, ng), bool)
                    if meta_diff.any():
                        lo = ug.min(-1)
                        rng = (ug.max(-1) - lo) / 3.0
                        ok = _near_e4m3_midpoint(lo) | _near_e4m3_midpoint(rng) | tok_c
                        assert ok[meta_diff].all(), "metadata differs away from an E4M3 rounding boundary"
                        bad_groups += int(meta_diff.sum())
                    code_diff = (gc != oc).reshape(n, ng, g) & ~meta_diff[..., None] & ~tok_c[..., None]
                    if code_diff.any():
                        s = F.e4m3_decode(os_)[..., None]
                        o = F.e4m3_decode(oo)[..., None]
                        qt = (ug - o) / np.where(s > 0, s, 1)
                        frac = np.abs(qt - np.floor(qt) - 0.5)
                        near = frac < 1e-3
                        step = np.abs(gc.reshape(n, ng, g).astype(int) - oc.reshape(n, ng, g).astype(int))
                        assert (near & (step == 1))[code_diff].all(), "code differs away from a rounding boundary"
                        bad_codes += int(code_diff.sum())
    rate = (bad_codes + bad_groups * g) / max(total, 1)
    assert rate <= max_rate, f"boundary mismatches too frequent: {rate:.2e}"
    return {"codes": total, "code_mismatch": bad_codes, "group_mismatch": bad_groups, "c_mismatch": c_diff}


def _build_both(case: Case, chunks, seq_start=None, anchor_is_base=True):
    """Append the same tokens (in the given chunk sizes) on both sides; return everything."""
    R32, R = rotation32(case.d, kind=case.rotation)
    gpu = GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    start = np.zeros(case.B, dtype=np.int64) if seq_start is None else np.array(seq_start)
    us = [None] * (case.P - 1)
    seed = case.seed
    for layer in range(case.L):
        for group in range(case.G):
            pos = start.copy()
            for ci, n in enumerate(chunks):
                kv_bf16, kv = kv_for(case, seed * 1000 + layer * 100 + group * 10 + ci, n, anchor_is_base)
                gpu.append(layer, group, kv_bf16, pos)
                comp = oracle.append(obuf, geom, R, layer, group, kv, pos, chained=case.chained,
                                     scaling=case.scaling, rotation=case.rotation)
                if layer == 0 and group == 0:
                    for j in range(case.P - 1):
                        us[j] = comp["u"][j] if us[j] is None else np.concatenate([us[j], comp["u"][j]], axis=-2)
                pos = pos + n
    st = gpu.status.cpu().numpy()
    assert st[1] == 0, "append reported a capacity overflow"
    return gpu, geom, obuf, R, us


@pytest.mark.parametrize("d,g", [(128, 32), (128, 16), (96, 32)])
def test_append_anchor_bitexact_and_residual_parity(d, g):
    case = Case(L=1, P=4, G=1, H=3, d=d, g=g, B=2, Nmax=320, seed=1)
    gpu, geom, obuf, R, us = _build_both(case, chunks=[200, 1, 37])
    gbuf = gpu.bytes_host()
    n = 238
    for b in range(case.B):
        for h in range(case.H):
            gv = plane_views(gbuf, geom, 0, 0, b, h)
            ov = plane_views(obuf, geom, 0, 0, b, h)
            for nm in ("AK", "AV"):
                assert np.array_equal(gv[nm], ov[nm]), f"anchor plane {nm} differs (b={b}, h={h})"
    stats = check_residual_parity(gbuf, obuf, geom, us, 0, 0, n, case.B, case.H)
    print("residual parity", stats)
    # the oracle takes the residual in the device's precision: every byte must match
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"


def test_append_ragged_starts():
    """Rows start at different positions (unaligned), appended in uneven chunks."""
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=3, Nmax=256, seed=2)
    gpu, geom, obuf, R, us = _build_both(case, chunks=[5, 1, 60], seq_start=[0, 3, 130])
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf[: geom.region_offset(0, 0, 0, 0)], obuf[: geom.region_offset(0, 0, 0, 0)])
    for b in range(case.B):
        for h in range(case.H):
            gv, ov = plane_views(gbuf, geom, 0, 0, b, h), plane_views(obuf, geom, 0, 0, b, h)
            assert np.array_equal(gv["AK"], ov["AK"]) and np.array_equal(gv["AV"], ov["AV"])


def test_append_exact_rotation_is_bitexact():
    """With R a signed permutation the rotation is exact in any precision, so
    every byte of every plane matches the float64 reading of the oracle too."""
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=2, Nmax=192, seed=3)
    rng = np.random.default_rng(7)
    perm = rng.permutation(128)
    Rp = np.zeros((128, 128), dtype=np.float32)
    Rp[np.arange(128), perm] = rng.choice([-1.0, 1.0], 128)
    gpu = GpuCache(case, Rp)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    kv_bf16, kv = kv_for(case, 11, 150)
    # keep only vectors whose residual x - c*a_hat is exact in float32 on the oracle side
    gpu.append(0, 0, kv_bf16, [0, 0])
    comp = oracle.append(obuf, geom, Rp.astype(np.float64), 0, 0, kv, [0, 0], precision="f64")
    gbuf = gpu.bytes_host()
    a_hat = oracle.dequantize(*comp["anchor"], 32)
    exact = np.ones((2, 2, 2, 150), bool)
    for j in range(3):
        cb = oracle.bf16_decode(comp["res"][j][3])[..., None]
        e = kv[j] - cb * a_hat
        exact &= np.all(e.astype(np.float32).astype(np.float64) == e, axis=-1)
    assert exact.mean() > 0.9
    for b in range(2):
        for h in range(2):
            for kvi in range(2):
                for j in range(3):
                    gc, gs, go, gcb = oracle.read_plane_tokens(gbuf, geom, 0, 0, b, h, kvi, "res", j, 150)
                    oc, os_, oo, ocb = oracle.read_plane_tokens(obuf, geom, 0, 0, b, h, kvi, "res", j, 150)
                    m = exact[kvi, b, h]
                    assert np.array_equal(gc[m], oc[m]) and np.array_equal(gs[m], os_[m])
                    assert np.array_equal(go[m], oo[m]) and np.array_equal(gcb, ocb)


def _queries(case, seed, loop):
    qb, q = synth.queries(seed * 7 + loop, case.B, case.H, case.d)
    kvb, kv = synth.looped_kv(seed * 13 + 1, case.workload(), batch=case.B, ntok=1)
    return qb, q, kvb[loop, 0, :, :, 0], kv[loop, 0, :, :, 0], kvb[loop, 1, :, :, 0], kv[loop, 1, :, :, 0]


@pytest.mark.parametrize("d,g,H,B,chained", [(128, 32, 2, 1, False), (128, 16, 3, 2, False),
                                             (96, 32, 5, 2, False), (96, 16, 2, 1, False),
                                             (128, 32, 2, 2, True), (96, 16, 3, 1, True)])
def test_decode_attention_matches_oracle(d, g, H, B, chained):
    """End to end: GPU-built cache + GPU attention against oracle cache + oracle
    attention; and the GPU kernel on the oracle's bytes (isolates the kernel)."""
    case = Case(L=2, P=4, G=1, H=H, d=d, g=g, B=B, Nmax=400, seed=4, chained=chained)
    n = 333
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[n])
    gbuf = gpu.bytes_host()
    scale = 1.0 / math.sqrt(d)
    seq = np.full(B, n)
    worst, worst_iso = 0.0, 0.0
    iso = GpuCache(case, rotation32(d)[0])
    iso.buf.copy_(torch.from_numpy(obuf))
    for layer in range(2):
        for loop in range(4):
            qb, q, kcb, kc, vcb, vc = _queries(case, layer + 10, loop)
            out = gpu.decode(layer, 0, loop, qb, kcb, vcb, seq, scale).cpu().numpy()
            ref = oracle.decode_attention(obuf, geom, R, layer, 0, loop, q, kc, vc, seq, scale,
                                          chained=chained)
            err = float(np.abs(out - ref).max())
            worst = max(worst, err)
            out_iso = iso.decode(layer, 0, loop, qb, kcb, vcb, seq, scale).cpu().numpy()
            worst_iso = max(worst_iso, float(np.abs(out_iso - ref).max()))
            assert err <= ATOL, f"layer {layer} loop {loop}: max abs err {err:.3e}"
    diff_bytes = int((gbuf != obuf).sum())
    print(f"worst max-abs error {worst:.3e} (kernel on oracle bytes {worst_iso:.3e}); "
          f"cache bytes differing {diff_bytes} of {obuf.size}")
    assert diff_bytes == 0
    assert worst_iso <= 1e-3   # 16-bit fixed-point query and value weights
    assert int(gpu.status.cpu()[0]) == 0


def test_decode_on_oracle_bytes_isolates_the_kernel():
    """Upload the oracle's cache bytes; the kernel must reproduce the oracle's attention
    over those exact bytes."""
    case = Case(L=1, P=4, G=1, H=4, d=128, g=32, B=2, Nmax=640, seed=5)
    R32, R = rotation32(128)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    kvb, kv = kv_for(case, 21, 600)
    oracle.append(obuf, geom, R, 0, 0, kv, [0, 0])
    gpu = GpuCache(case, R32)
    gpu.buf.copy_(torch.from_numpy(obuf))
    seq = np.array([600, 517])
    worst = 0.0
    for loop in range(4):
        qb, q, kcb, kc, vcb, vc = _queries(case, 3, loop)
        out = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, 0.0883883476).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kc, vc, seq, 0.0883883476)
        worst = max(worst, float(np.abs(out - ref).max()))
    assert worst <= 1e-3, worst   # 16-bit fixed-point query and value weights


@pytest.mark.parametrize("seq", [[0, 1, 63, 64], [65, 127, 128, 129], [1, 0, 0, 200]])
def test_decode_ragged_and_empty(seq):
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=4, Nmax=256, seed=6)
    R32, R = rotation32(128)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    kvb, kv = kv_for(case, 31, 200)
    oracle.append(obuf, geom, R, 0, 0, kv, [0, 0, 0, 0])
    gpu = GpuCache(case, R32)
    gpu.buf.copy_(torch.from_numpy(obuf))
    seq = np.array(seq)
    for loop in (0, 3):
        qb, q, kcb, kc, vcb, vc = _queries(case, 5, loop)
        out = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, 0.09).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kc, vc, seq, 0.09)
        assert np.abs(out - ref).max() <= 1e-3
    # an empty row returns the current token's value exactly
    for b in np.nonzero(seq == 0)[0]:
        assert np.array_equal(out[b], vc[b].astype(np.float32))


def test_decode_repeated_calls_reuse_workspace():
    """The same call twice on one workspace gives the same bits and a clear status word."""
    case = Case(L=1, P=4, G=1, H=3, d=128, g=32, B=2, Nmax=2048, seed=7)
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[1500])
    qb, q, kcb, kc, vcb, vc = _queries(case, 9, 1)
    a = gpu.decode(0, 0, 1, qb, kcb, vcb, [1500, 1500], 0.08)
    b = gpu.decode(0, 0, 1, qb, kcb, vcb, [1500, 1500], 0.08)
    assert torch.equal(a, b)
    assert gpu.status.tolist() == [0, 0, 0, 0]


def test_bf16_comparator_matches_softmax_attention():
    import decode_attention_rq_gb300 as rq
    rng = np.random.default_rng(8)
    for d in (128, 96):
        B, H, S = 3, 4, 300
        seq = np.array([300, 1, 0])
        k = torch.from_numpy(rng.standard_normal((B, H, S, d), dtype=np.float32)).to(torch.bfloat16)
        v = torch.from_numpy(rng.standard_normal((B, H, S, d), dtype=np.float32)).to(torch.bfloat16)
        q = torch.from_numpy(rng.standard_normal((B, H, d), dtype=np.float32)).to(torch.bfloat16)
        kc = torch.from_numpy(rng.standard_normal((B, H, d), dtype=np.float32)).to(torch.bfloat16)
        vc = torch.from_numpy(rng.standard_normal((B, H, d), dtype=np.float32)).to(torch.bfloat16)
        dev = "cuda:0"
        ws_bytes = rq.rq_bf16_workspace_bytes(B, H, d)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
        sl = torch.as_tensor(seq.astype(np.int32), device=dev)
        scale = 1 / math.sqrt(d)
        rq.rq_decode_attention_bf16(k.to(dev), v.to(dev), kc.to(dev), vc.to(dev), q.to(dev), sl, B, H, d, S,
                                    scale, out, ws, ws_bytes)
        o = out.cpu().numpy()
        K, V, Q = k.double().numpy(), v.double().numpy(), q.double().numpy()
        KC, VC = kc.double().numpy(), vc.double().numpy()
        for b in range(B):
            for h in range(H):
                n = seq[b]
                ref = oracle.attention(Q[b, h], np.concatenate([K[b, h, :n], KC[b, h][None]]),
                                       np.concatenate([V[b, h, :n], VC[b, h][None]]), scale)
                assert np.abs(o[b, h] - ref).max() <= 1e-4


def test_chained_append_bitexact():
    """Chained mode: each loop coded against the rebuilt next loop; every byte matches."""
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=2, Nmax=256, seed=9, chained=True)
    gpu, geom, obuf, R, us = _build_both(case, chunks=[130, 3])
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"


@pytest.mark.parametrize("P,d", [(8, 128), (16, 96)])
def test_large_loop_groups_shared(P, d):
    """Groups of 8 and 16 loops per anchor (shared anchor): every byte matches the
    oracle's, and loops across the group decode within tolerance (each residual
    loop reads the anchor and its own plane, whatever the group length)."""
    import decode_attention_rq_gb300 as rq
    case = Case(L=1, P=P, G=2, H=2, d=d, g=32, B=2, Nmax=200, seed=12 + P)
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[170, 1], anchor_is_base=False)
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    seq = np.array([171, 90])
    scale = 1 / math.sqrt(d)
    worst = 0.0
    for group in (0, 1):
        for loop in (0, P // 2, P - 2, P - 1):
            qb, q, kcb, kc, vcb, vc = _queries(case, 40 + group, loop)
            out = gpu.decode(0, group, loop, qb, kcb, vcb, seq, scale).cpu().numpy()
            ref = oracle.decode_attention(obuf, geom, R, 0, group, loop, q, kc, vc, seq, scale)
            err = float(np.abs(out - ref).max())
            worst = max(worst, err)
            assert err <= ATOL, f"P={P} group {group} loop {loop}: max abs err {err:.3e}"
    assert int(gpu.status.cpu()[0]) == 0
    print(f"P={P}: worst max-abs error {worst:.3e}; cache bytes equal")


@pytest.mark.parametrize("d,g", [(128, 32), (96, 16)])
def test_large_chained_groups(d, g):
    """Chained groups of 8 loops: appends (each loop coded against the rebuilt
    next one) match byte for byte; every loop decodes within 2e-3 (loop 0 reads
    the anchor and seven residual planes).  Chained groups of 16 loops are
    refused with UNSUPPORTED (a call would read fifteen planes)."""
    import decode_attention_rq_gb300 as rq
    case = Case(L=1, P=8, G=1, H=2, d=d, g=g, B=2, Nmax=192, seed=21, chained=True)
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[130, 1], anchor_is_base=False)
    assert np.array_equal(gpu.bytes_host(), obuf)
    seq = np.array([131, 70])
    scale = 1 / math.sqrt(d)
    worst = 0.0
    for loop in (0, 3, 6, 7):
        qb, q, kcb, kc, vcb, vc = _queries(case, 50, loop)
        out = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, scale).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kc, vc, seq, scale, chained=True)
        err = float(np.abs(out - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"loop {loop}: max abs err {err:.3e}"
    assert gpu.status.tolist() == [0, 0, 0, 0]
    print(f"chained P=8 d={d} g={g}: worst max-abs error {worst:.3e}; cache bytes equal")
    big = GpuCache(Case(L=1, P=16, G=1, H=2, d=d, g=g, B=1, Nmax=64, seed=22, chained=True), rotation32(d)[0])
    qb, q, kcb, kc, vcb, vc = _queries(case, 51, 0)
    with pytest.raises(rq.RqError) as e:
        big.decode(0, 0, 0, qb[:1], kcb[:1], vcb[:1], np.array([10]), 0.1, batch=1)
    assert e.value.status == 6   # RQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("chained", [False, True])
def test_norm_ratio_scaling(chained):
    """Norm-ratio coefficient (||x|| / ||ref||, the appendix alternative to least
    squares): every cache byte equals the oracle's, and decode (unchanged: it uses
    the stored coefficient) stays within tolerance."""
    case = Case(L=1, P=4, G=1, H=3, d=128, g=32, B=2, Nmax=256, seed=31, chained=chained, scaling="norm")
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[200, 1])
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    seq = np.array([201, 150])
    for loop in range(4):
        qb, q, kcb, kc, vcb, vc = _queries(case, 60, loop)
        out = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, 1 / math.sqrt(128)).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kc, vc, seq, 1 / math.sqrt(128),
                                      chained=chained)
        assert np.abs(out - ref).max() <= ATOL


def test_walsh_hadamard_rotation():
    """A normalised Walsh-Hadamard matrix as R (Sylvester construction, d = 128): the
    library takes any orthogonal R as a dense matrix, so the same append and decode
    paths must match the oracle run with the same binary32 R."""
    import decode_attention_rq_gb300 as rq
    d = 128
    Hm = np.array([[1.0]])
    while Hm.shape[0] < d:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    R32 = (Hm / np.sqrt(d)).astype(np.float32)
    R = R32.astype(np.float64)
    assert np.abs(R @ R.T - np.eye(d)).max() < 1e-6
    case = Case(L=1, P=4, G=1, H=2, d=d, g=32, B=2, Nmax=192, seed=33)
    gpu = GpuCache(case, R32)
    geom = _geom(case)
    obuf = np.zeros(geom.total_bytes, dtype=np.uint8)
    kv_bf16, kv = kv_for(case, 3301, 150)
    start = np.zeros(case.B, dtype=np.int64)
    gpu.append(0, 0, kv_bf16, start)
    oracle.append(obuf, geom, R, 0, 0, kv, start)
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    seq = np.array([150, 77])
    for loop in range(4):
        qb, q, kcb, kc, vcb, vc = _queries(case, 70, loop)
        out = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, 1 / math.sqrt(d)).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kc, vc, seq, 1 / math.sqrt(d))
        assert np.abs(out - ref).max() <= ATOL


@pytest.mark.parametrize("chained", [False, True])
def test_hadamard_mode_fast_transform(chained):
    """RQ_MODE_HADAMARD: no R on the device; the append, the query prep and the
    merge run the fast Walsh-Hadamard transform.  Every cache byte equals the
    oracle's (whose binary32 path follows the same butterfly order), every loop
    decodes within 2e-3 of the oracle attention over those bytes."""
    case = Case(L=1, P=4, G=1, H=3, d=128, g=32, B=2, Nmax=256, seed=34, chained=chained, rotation="hadamard")
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[190, 1, 9])
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf), f"{int((gbuf != obuf).sum())} cache bytes differ"
    seq = np.array([200, 131])
    worst = 0.0
    for loop in range(4):
        qb, q, kcb, kc, vcb, vc = _queries(case, 80, loop)
        out = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, 1 / math.sqrt(128)).cpu().numpy()
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kc, vc, seq, 1 / math.sqrt(128),
                                      chained=chained)
        err = float(np.abs(out - ref).max())
        worst = max(worst, err)
        assert err <= ATOL, f"loop {loop}: max abs err {err:.3e}"
    assert gpu.status.tolist() == [0, 0, 0, 0]
    print(f"hadamard chained={chained}: worst max-abs error {worst:.3e}; cache bytes equal")


def test_huginn_groups_and_layers():
    """Several loop groups and layers: regions do not overlap, each group decodes right."""
    case = Case(L=2, P=4, G=3, H=3, d=96, g=32, B=2, Nmax=192, seed=10)
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[150], anchor_is_base=False)
    gbuf = gpu.bytes_host()
    assert np.array_equal(gbuf, obuf)
    seq = np.array([150, 97])
    for layer, group in [(0, 0), (1, 2), (0, 1)]:
        for loop in (0, 3):
            qb, q, kcb, kc, vcb, vc = _queries(case, layer * 3 + group, loop)
            out = gpu.decode(layer, group, loop, qb, kcb, vcb, seq, 1 / math.sqrt(96)).cpu().numpy()
            ref = oracle.decode_attention(obuf, geom, R, layer, group, loop, q, kc, vc, seq, 1 / math.sqrt(96))
            assert np.abs(out - ref).max() <= ATOL


@pytest.mark.parametrize("d,g", [(128, 32), (96, 16)])
def test_residual_codes_against_the_float64_reading(d, g):
    """The same random data against the oracle's float64 rotation (e = x - c a_hat
    and u = R e without binary32 rounding): this check does not depend on the
    device's summation order.  Anchor planes and coefficients are bit-exact; the
    residual codes and metadata obey the boundary rule (check_residual_parity)."""
    case = Case(L=1, P=4, G=1, H=3, d=d, g=g, B=2, Nmax=320, seed=13)
    R32, R = rotation32(d)
    gpu = GpuCache(case, R32)
    geom = _geom(case)
    ob64 = np.zeros(geom.total_bytes, dtype=np.uint8)
    n = 300
    kvb, kv = kv_for(case, 1301, n)
    start = np.zeros(case.B, dtype=np.int64)
    gpu.append(0, 0, kvb, start)
    comp = oracle.append(ob64, geom, R, 0, 0, kv, start, precision="f64")
    gbuf = gpu.bytes_host()
    for b in range(case.B):
        for h in range(case.H):
            gv, ov = plane_views(gbuf, geom, 0, 0, b, h), plane_views(ob64, geom, 0, 0, b, h)
            for nm in ("AK", "AV"):
                assert np.array_equal(gv[nm], ov[nm]), f"anchor plane {nm} differs (b={b}, h={h})"
    stats = check_residual_parity(gbuf, ob64, geom, comp["u"], 0, 0, n, case.B, case.H)
    print(f"d={d} g={g} against the float64 reading: {stats}")


@pytest.mark.parametrize("chained", [False, True])
def test_decode_with_many_partials_per_head(chained):
    """Long rows at batch 1: every 128-token unit has its own decode CTA, so each
    (row, head) has 24 partial states and the merge combines them in two
    batches.  Every loop within 2e-3 of the oracle; repeated calls equal."""
    case = Case(L=1, P=4, G=1, H=2, d=128, g=32, B=1, Nmax=3200, seed=19, chained=chained)
    n = 3050                                   # 24 units: 23 full, one of 106 tokens
    gpu, geom, obuf, R, _ = _build_both(case, chunks=[n])
    assert np.array_equal(gpu.bytes_host(), obuf)
    scale = 1.0 / math.sqrt(128)
    seq = np.full(1, n)
    for loop in range(4):
        qb, q, kcb, kc, vcb, vc = _queries(case, 20, loop)
        out = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, scale)
        again = gpu.decode(0, 0, loop, qb, kcb, vcb, seq, scale)
        assert torch.equal(out, again)
        ref = oracle.decode_attention(obuf, geom, R, 0, 0, loop, q, kc, vc, seq, scale, chained=chained)
        err = float(np.abs(out.cpu().numpy() - ref).max())
        assert err <= ATOL, f"loop {loop}: max abs err {err:.3e}"
    assert gpu.status.tolist() == [0, 0, 0, 0]

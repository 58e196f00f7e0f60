"""Pins for the oracle's cache layout and storage accounting (no GPU)."""
import json
import os

import numpy as np
import pytest

import synth
import oracle
from oracle import layout as Lo
from oracle import method as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "storage_accounting.json")


def test_storage_accounting_reproduces_the_pages():
    gold = {e["quantity"].split(" (")[0]: e for e in json.load(open(GOLDEN))["entries"]}
    acc = Lo.bits_per_element(128, 32, 4)
    got = {
        "uncompressed bits per KV element position over the 4 loops": acc["bf16"],
        "code bits per element position over the 4 loops": 4 + 2 * 3,
        "compression ratio before metadata": acc["codes_only_ratio"],
        "compression ratio with FP8 scale+offset per group and one BF16 coefficient per residual vector": acc["ratio"],
        "theoretical KV storage reduction vs BF16, percent": 100 * acc["reduction"],
    }
    for k, e in gold.items():
        assert abs(got[k] - e["value"]) <= e["tolerance"], (k, got[k], e["value"])
    # closed form: 4.5 + 3 x 2.625 = 12.375 bits
    assert acc["anchor"] == 4.5 and acc["residual"] == 2.625 and acc["total"] == 12.375


def test_storage_other_shapes():
    assert Lo.bits_per_element(128, 16, 4)["total"] == 14.375
    assert Lo.bits_per_element(96, 32, 4)["total"] == 4.5 + 3 * (2 + 0.5 + 16 / 96)


@pytest.mark.parametrize("P", [8, 16])
def test_storage_of_larger_loop_groups(P):
    """Groups of 8 or 16 loops per anchor (the appendix variant): one INT4 anchor and
    P-1 INT2 residuals.  Closed form from the record sizes at d=128, g=32: anchor
    4 + 16/32 bits, each residual 2 + 16/32 + 16/128 bits per element."""
    acc = Lo.bits_per_element(128, 32, P)
    assert acc["total"] == pytest.approx(4.5 + (P - 1) * 2.625)
    assert acc["reduction"] == pytest.approx(1 - (4.5 + (P - 1) * 2.625) / (16 * P))
    geom = Lo.Geometry(1, P, 1, 1, 128, 32, 1, 64)
    # one tile of 64 tokens, K and V: bytes = 64 tokens x 128 channels x bits / 8
    assert geom.region == 2 * 64 * 128 * acc["total"] / 8


@pytest.mark.parametrize("d,g,per_token", [(128, 32, 396), (128, 16, 2 * 80 + 6 * 50), (96, 32, 2 * 54 + 6 * 32)])
def test_geometry_bytes_match_the_accounting(d, g, per_token):
    geom = Lo.Geometry(1, 4, 1, 1, d, g, 1, 640)
    assert geom.region == 10 * per_token * 64          # 10 tiles of 64 tokens
    assert geom.region * 8 / (640 * 2 * d) == Lo.bits_per_element(d, g, 4)["total"]
    for sz in (geom.a_tile, geom.r_tile, geom.a_codes, geom.r_codes, geom.meta):
        assert sz % 16 == 0


def _small_cache(chained, seed=0, n=150, B=2, H=3, d=128, g=32):
    w = synth.Workload("t", 2, 4, 2, H, d, g, B, n, synth.OURO_ALPHAS, True)
    geom = Lo.Geometry(2, 4, 2, H, d, g, B, 200)
    buf = np.zeros(geom.total_bytes, dtype=np.uint8)
    R = synth.rotation(d).astype(np.float32).astype(np.float64)
    _, kv = synth.looped_kv(seed, w, batch=B, ntok=n)
    comps = []
    # write in two appends (prefill then a few more tokens) to layer 1, group 1
    comps.append(oracle.append(buf, geom, R, 1, 1, kv[..., :100, :], [0] * B, chained))
    comps.append(oracle.append(buf, geom, R, 1, 1, kv[..., 100:, :], [100] * B, chained))
    return geom, buf, R, kv, comps


@pytest.mark.parametrize("chained", [False, True])
def test_pack_read_roundtrip_and_reconstruction(chained):
    geom, buf, R, kv, comps = _small_cache(chained)
    recon = np.concatenate([c["recon"] for c in comps], axis=-2)       # [P,2,B,H,n,d]
    for b in range(2):
        for h in range(3):
            for loop in range(4):
                K, V = oracle.reconstruct(buf, geom, R, 1, 1, b, h, loop, 150, chained)
                assert np.array_equal(K, recon[loop, 0, b, h])
                assert np.array_equal(V, recon[loop, 1, b, h])
    # other (layer, group) regions untouched
    off = geom.region_offset(1, 1, 0, 0)
    assert not buf[:off].any()


def test_code_positions_in_bytes():
    """Spot-check the documented bit positions against hand-built bytes."""
    geom = Lo.Geometry(1, 4, 1, 1, 128, 32, 1, 64)
    buf = np.zeros(geom.total_bytes, dtype=np.uint8)
    codes4 = np.zeros((1, 128), dtype=np.uint8)
    codes4[0, 0], codes4[0, 1], codes4[0, 5] = 3, 12, 7
    addr, sh = Lo._code_addresses(geom, 0, geom.a_tile, np.array([5]), 4, channel_major=False)
    Lo._write_codes(buf, addr, sh, codes4, 4)
    row = 5 * 64
    assert buf[row] == 3 | (12 << 4) and buf[row + 2] == 7 << 4
    buf[:] = 0
    addr, sh = Lo._code_addresses(geom, 0, geom.a_tile, np.array([5]), 4, channel_major=True)
    Lo._write_codes(buf, addr, sh, codes4, 4)
    # channel-major: channel 1's row is bytes 32..63; token 5 is token 5 of word 0:
    # byte 5 mod 4 = 1, high nibble
    assert buf[32 + 1] == 12 << 4 and buf[0 + 1] == 3 << 4 and buf[5 * 32 + 1] == 7 << 4
    buf[:] = 0
    codes2 = np.zeros((1, 128), dtype=np.uint8)
    codes2[0, 6] = 2
    base = geom.res_plane(0, 1)
    addr, sh = Lo._code_addresses(geom, base, geom.r_tile, np.array([7]), 2, channel_major=True)
    Lo._write_codes(buf, addr, sh, codes2, 2)
    assert buf[base + 6 * 16 + 3] == 2 << 2      # token 7 of word 0: byte 3, bits 2-3


@pytest.mark.parametrize("bits", [4, 2])
def test_channel_major_masks_give_consecutive_tokens(bits):
    """The documented V word order: each byte mask of a 32-bit word leaves four
    consecutive tokens of the channel, token t0+i in byte i."""
    geom = Lo.Geometry(1, 2, 1, 1, 128, 32, 1, 64)
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 1 << bits, size=(64, 128), dtype=np.uint8)
    buf = np.zeros(geom.total_bytes, dtype=np.uint8)
    tile = geom.a_tile if bits == 4 else geom.r_tile
    base = geom.anchor_plane(1) if bits == 4 else geom.res_plane(0, 1)
    addr, sh = Lo._code_addresses(geom, base, tile, np.arange(64), bits, channel_major=True)
    Lo._write_codes(buf, addr, sh, codes, bits)
    row_bytes = 64 * bits // 8
    masks = [0x0F0F0F0F, 0xF0F0F0F0] if bits == 4 else [0x03030303 << (2 * m) for m in range(4)]
    for ch in (0, 1, 77, 127):
        words = buf[base + ch * row_bytes: base + (ch + 1) * row_bytes].view("<u4")
        t0 = 0
        for w in words:
            for k, mk in enumerate(masks):
                got = [((int(w) & mk) >> (8 * i + k * bits)) & ((1 << bits) - 1) for i in range(4)]
                assert got == list(codes[t0:t0 + 4, ch]), (ch, t0)
                t0 += 4
        assert t0 == 64


@pytest.mark.parametrize("chained", [False, True])
def test_read_counts_shared_vs_chained(chained, monkeypatch):
    """Shared anchor: a loop reads the anchor plane and its own residual plane
    (2 reads); chained: the anchor plus every residual plane down to the loop,
    4 reads for the farthest loop of 4 ([EXPL] shared-master paragraph)."""
    geom, buf, R, kv, comps = _small_cache(chained)
    reads = []
    orig = oracle.read_plane_tokens

    def spy(*a, **k):
        reads.append(a[7])
        return orig(*a, **k)
    monkeypatch.setattr(oracle, "read_plane_tokens", spy)
    for loop, want_chained in [(0, 4), (1, 3), (2, 2), (3, 1)]:
        reads.clear()
        oracle.reconstruct(buf, geom, R, 1, 1, 0, 0, loop, 150, chained)
        per_kv = len(reads) // 2
        assert per_kv == (want_chained if chained else (2 if loop < 3 else 1))


def test_decode_attention_over_cache():
    geom, buf, R, kv, comps = _small_cache(False, n=150)
    recon = np.concatenate([c["recon"] for c in comps], axis=-2)
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 3, 128))
    kc = rng.standard_normal((2, 3, 128))
    vc = rng.standard_normal((2, 3, 128))
    seq = np.array([150, 37])
    out = oracle.decode_attention(buf, geom, R, 1, 1, 2, q, kc, vc, seq, 0.0883883)
    for b in range(2):
        for h in range(3):
            n = seq[b]
            K = np.concatenate([recon[2, 0, b, h, :n], kc[b, h][None]])
            V = np.concatenate([recon[2, 1, b, h, :n], vc[b, h][None]])
            assert np.allclose(out[b, h], M.attention(q[b, h], K, V, 0.0883883), rtol=0, atol=1e-13)
    # an empty cache attends to the current token only
    out0 = oracle.decode_attention(buf, geom, R, 1, 1, 0, q, kc, vc, np.array([0, 0]), 0.1)
    assert np.array_equal(out0, vc)


@pytest.mark.parametrize("chained", [False, True])
def test_decode_attention_append_writes_the_next_slot(chained):
    """The last-loop call followed by the token's append: the output is the
    attention over the cache as it was; the token of every loop then reads back
    from slot seq_lens[b] within its quantization error (a wrong slot reads
    zeros, a wrong plane another loop); earlier slots and the next slot keep
    their bytes; a row with one free slot fills it; a row at capacity is
    attended but left untouched."""
    d, g, H, B, P, cap = 64, 32, 2, 4, 4, 128
    geom = Lo.Geometry(1, P, 1, H, d, g, B, cap)
    R = synth.rotation(d).astype(np.float32).astype(np.float64)
    w = synth.Workload("t", 1, P, 1, H, d, g, B, cap, synth.OURO_ALPHAS, True)
    _, kv = synth.looped_kv(5, w, batch=B, ntok=100)
    buf = np.zeros(geom.total_bytes, dtype=np.uint8)
    oracle.append(buf, geom, R, 0, 0, kv, [0, 0, 28, 27], chained)  # row 2 full, row 3 one slot short
    before = buf.copy()
    _, cur = synth.looped_kv(6, w, batch=B, ntok=1)
    kv_cur = cur[..., 0, :]                                          # [P, 2, B, H, d]
    q = np.random.default_rng(8).standard_normal((B, H, d))
    seq = np.array([100, 37, cap, cap - 1])
    out, ok = oracle.decode_attention_append(buf, geom, R, 0, 0, q, kv_cur, seq, 0.125, chained=chained)
    assert ok.tolist() == [True, True, False, True]
    ref = oracle.decode_attention(before, geom, R, 0, 0, P - 1, q, kv_cur[P - 1, 0], kv_cur[P - 1, 1], seq, 0.125,
                                  chained=chained)
    assert np.array_equal(out, ref)
    r2 = geom.region_offset(0, 0, 2, 0)
    assert np.array_equal(buf[r2:r2 + H * geom.region], before[r2:r2 + H * geom.region])
    # what compressing the token alone gives (its reconstruction per loop)
    recon = M.compress_group(kv_cur[..., None, :], R, g, chained=chained)["recon"][..., 0, :]
    worst = {}
    for b in (0, 1, 3):
        n = int(seq[b])
        m = min(n + 2, cap)
        for h in range(H):
            for loop in range(P):
                K0, V0 = oracle.reconstruct(before, geom, R, 0, 0, b, h, loop, m, chained)
                K1, V1 = oracle.reconstruct(buf, geom, R, 0, 0, b, h, loop, m, chained)
                for kvi, (X0, X1) in enumerate(((K0, K1), (V0, V1))):
                    assert np.array_equal(X1[:n], X0[:n])                 # earlier slots unchanged
                    if n + 1 < cap:
                        assert np.array_equal(X1[n + 1], X0[n + 1])      # the next slot too
                    assert np.array_equal(X1[n], recon[loop, kvi, b, h])    # this slot, this plane
                    x = kv_cur[loop, kvi, b, h]
                    rel = np.linalg.norm(X1[n] - x) / np.linalg.norm(x)
                    worst[loop] = max(worst.get(loop, 0.0), rel)
    print("relative reconstruction error of the appended token per loop", worst)
    assert all(v < 0.25 for v in worst.values())


def test_paged_pool_moves_whole_tiles():
    """The paged view holds every mapped tile byte for byte at its page (a page =
    one 64-token block of every plane of every head: 396 B x 64 x H at d = 128,
    g = 32, 4 loops); unmapped pages stay zero; reading the pool back through
    the table gives the contiguous cache again."""
    geom, buf, R, kv, comps = _small_cache(False)          # 2 layers, 2 groups, B = 2, H = 3, 200 slots
    ntiles = geom.ntiles
    num_pages = 2 * ntiles + 2
    rng = np.random.default_rng(4)
    perm = rng.permutation(num_pages)
    table = perm[: 2 * ntiles].reshape(2, ntiles)
    pool = Lo.paged_pool(buf, geom, table, num_pages)
    head_block = 396 * 64
    page_bytes = 3 * head_block
    assert pool.size == 2 * 2 * num_pages * page_bytes
    # unmapped pages are zero
    for lg in range(4):
        for p in perm[2 * ntiles:]:
            o = (lg * num_pages + p) * page_bytes
            assert not pool[o:o + page_bytes].any()
    # back through the table: every region equals the contiguous one
    back = np.zeros_like(buf)
    for layer in range(2):
        for group in range(2):
            for b in range(2):
                for h in range(3):
                    r0 = geom.region_offset(layer, group, b, h)
                    for t in range(ntiles):
                        src = ((layer * 2 + group) * num_pages + table[b, t]) * page_bytes + h * head_block
                        off = 0
                        for plane, tb in [(geom.anchor_plane(0), geom.a_tile), (geom.anchor_plane(1), geom.a_tile)] + \
                                [(geom.res_plane(j, kv_), geom.r_tile) for j in range(3) for kv_ in (0, 1)]:
                            back[r0 + plane + t * tb: r0 + plane + (t + 1) * tb] = pool[src + off: src + off + tb]
                            off += tb
                    assert off == head_block
    assert np.array_equal(back, buf)


def test_grouped_query_attention_is_multi_head_over_copied_kv_heads():
    """Grouped-query reading: query head qh attends with KV head qh // (Hq / H).
    Pinned against multi-head attention over a cache whose heads are copies
    (head qh of the copy = KV head qh // 2): the outputs are identical, and a
    mapping like qh % H would fail."""
    H, Hq, d, g, B = 2, 4, 64, 32, 2
    geom = Lo.Geometry(1, 4, 1, H, d, g, B, 96)
    geom_mha = Lo.Geometry(1, 4, 1, Hq, d, g, B, 96)
    R = synth.rotation(d).astype(np.float32).astype(np.float64)
    w = synth.Workload("t", 1, 4, 1, H, d, g, B, 96, synth.OURO_ALPHAS, True)
    _, kv = synth.looped_kv(9, w, batch=B, ntok=70)                   # [P, 2, B, H, n, d]
    buf = np.zeros(geom.total_bytes, dtype=np.uint8)
    oracle.append(buf, geom, R, 0, 0, kv, [0, 0])
    buf_mha = np.zeros(geom_mha.total_bytes, dtype=np.uint8)
    oracle.append(buf_mha, geom_mha, R, 0, 0, np.repeat(kv, 2, axis=3), [0, 0])
    buf_tiled = np.zeros(geom_mha.total_bytes, dtype=np.uint8)        # head qh = KV head qh % H
    oracle.append(buf_tiled, geom_mha, R, 0, 0, np.tile(kv, (1, 1, 1, 2, 1, 1)), [0, 0])
    rng = np.random.default_rng(2)
    q = rng.standard_normal((B, Hq, d))
    kc, vc = rng.standard_normal((B, H, d)), rng.standard_normal((B, H, d))
    seq = np.array([70, 41])
    for loop in (0, 3):
        out = oracle.decode_attention(buf, geom, R, 0, 0, loop, q, kc, vc, seq, 0.125)
        ref = oracle.decode_attention(buf_mha, geom_mha, R, 0, 0, loop, q, np.repeat(kc, 2, axis=1),
                                      np.repeat(vc, 2, axis=1), seq, 0.125)
        assert np.array_equal(out, ref)
        wrong = oracle.decode_attention(buf_tiled, geom_mha, R, 0, 0, loop, q, np.tile(kc, (1, 2, 1)),
                                        np.tile(vc, (1, 2, 1)), seq, 0.125)
        assert not np.allclose(out, wrong)

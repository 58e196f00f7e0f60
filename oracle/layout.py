"""Byte layout of the compressed cache, written independently of the device code (oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The pages fix what is stored per vector -- INT4 anchor codes, INT2
residual codes per earlier loop, an FP8 scale and offset per channel group,
one BF16 coefficient per residual vector ([EXPL] worked storage example;
[SUMM] main-results paragraph on effective bit width) -- but not where the
bytes go.  The format below is this library's, stated in include/rq.h; the
oracle writes and reads it from that statement alone.

Hierarchy:  cache = [layer][loop group][batch row][head] regions.
Region  = plane AK, plane AV, then for j = 0 .. P-2: plane RK_j, plane RV_j.
Plane   = ceil(max_seq_len / 64) tiles of 64 token slots, tile t holding
          positions 64t .. 64t+63.
Anchor tile   = codes (64 * d/2 bytes) | meta (64 * ng * 2 bytes)
Residual tile = codes (64 * d/4 bytes) | meta (64 * ng * 2 bytes) | c (64 * 2 bytes)
Codes of K planes are token-major: row r (64 rows) holds the token's d
  codes, 4-bit: byte i = ch 2i (bits 0-3) | ch 2i+1 (bits 4-7);
  2-bit: byte i = ch 4i+m at bits 2m..2m+1, m = 0..3.
Codes of V planes are channel-major: row ch (d rows) holds the 64 tokens'
  codes of that channel in 32-bit words; 4-bit: word w (8 tokens) has in byte
  i token 8w+i (bits 0-3) and token 8w+4+i (bits 4-7); 2-bit: word j (16
  tokens) has in byte i token 16j+4m+i at bits 2m..2m+1, m = 0..3.  (Masking
  a word with 0x0F0F0F0F, 0xF0F0F0F0 or 0x03030303 << 2m leaves four
  consecutive tokens, one per byte.)
Meta: row r holds, for each group i, the E4M3 scale byte then the E4M3
  offset byte.  c: BF16 little-endian, slot r.
Every tile size is a multiple of 16 bytes (64 rows), so every tile, and
every sub-block of it, starts 16-byte aligned when the buffer does.
"""
from __future__ import annotations

import dataclasses

import numpy as np

TILE = 64

__all__ = ["TILE", "Geometry", "pack_group", "read_plane_tokens", "bits_per_element"]


@dataclasses.dataclass(frozen=True)
class Geometry:
    num_layers: int
    loops_per_group: int
    num_groups: int
    num_heads: int
    head_dim: int
    group_size: int
    max_batch: int
    max_seq_len: int

    @property
    def ng(self) -> int:
        return self.head_dim // self.group_size

    @property
    def ntiles(self) -> int:
        return -(-self.max_seq_len // TILE)

    # per-tile sub-block sizes, bytes
    @property
    def a_codes(self) -> int:
        return TILE * self.head_dim // 2

    @property
    def r_codes(self) -> int:
        return TILE * self.head_dim // 4

    @property
    def meta(self) -> int:
        return TILE * self.ng * 2

    @property
    def a_tile(self) -> int:
        return self.a_codes + self.meta

    @property
    def r_tile(self) -> int:
        return self.r_codes + self.meta + TILE * 2

    @property
    def region(self) -> int:
        n = self.ntiles
        return 2 * n * self.a_tile + 2 * (self.loops_per_group - 1) * n * self.r_tile

    @property
    def total_bytes(self) -> int:
        return (self.num_layers * self.num_groups * self.max_batch * self.num_heads) * self.region

    def region_offset(self, layer: int, group: int, b: int, h: int) -> int:
        idx = ((layer * self.num_groups + group) * self.max_batch + b) * self.num_heads + h
        return idx * self.region

    def anchor_plane(self, kv: int) -> int:
        return kv * self.ntiles * self.a_tile

    def res_plane(self, j: int, kv: int) -> int:
        return 2 * self.ntiles * self.a_tile + (2 * j + kv) * self.ntiles * self.r_tile


def paged_pool(buf: np.ndarray, geom: Geometry, table: np.ndarray, num_pages: int) -> np.ndarray:
    """The paged layout's pool holding the same cache as the contiguous bytes buf.

    Paged layout (a block table, as a paged serving engine lays out its KV cache;
    the pages integrate the method into such an engine): each (layer, group)
    owns num_pages pages; page p holds, for every head h in order, the tiles
    of one 64-token block of every plane -- anchor K, anchor V, then residual
    plane j's K and V for j = 0 .. P-2 -- each tile byte for byte as in the
    contiguous plane.  Tile t of batch row b is in page table[b, t]; entries
    below 0 map nothing.  Pages no (row, tile) maps to stay zero."""
    P, H = geom.loops_per_group, geom.num_heads
    planes = [(geom.anchor_plane(0), geom.a_tile), (geom.anchor_plane(1), geom.a_tile)]
    for j in range(P - 1):
        planes += [(geom.res_plane(j, 0), geom.r_tile), (geom.res_plane(j, 1), geom.r_tile)]
    head_block = sum(tb for _, tb in planes)
    page_bytes = H * head_block
    L, G = geom.num_layers, geom.num_groups
    pool = np.zeros(L * G * num_pages * page_bytes, dtype=np.uint8)
    table = np.asarray(table)
    for layer in range(L):
        for group in range(G):
            for b in range(table.shape[0]):
                for t in range(min(table.shape[1], geom.ntiles)):
                    page = int(table[b, t])
                    if page < 0:
                        continue
                    for h in range(H):
                        dst = ((layer * G + group) * num_pages + page) * page_bytes + h * head_block
                        src_region = geom.region_offset(layer, group, b, h)
                        for plane_base, tb in planes:
                            src = src_region + plane_base + t * tb
                            pool[dst:dst + tb] = buf[src:src + tb]
                            dst += tb
    return pool


def _code_addresses(geom: Geometry, plane_base: int, tile_bytes: int, pos: np.ndarray,
                    bits: int, channel_major: bool):
    """Byte address and bit shift of every (token, channel) code.

    pos: int64 [n] token positions.  Returns (addr [n, d], shift [n, d])."""
    d = geom.head_dim
    per_byte = 8 // bits
    t, r = np.divmod(pos, TILE)
    tile_base = plane_base + t * tile_bytes                    # [n]
    ch = np.arange(d)
    if channel_major:
        row_bytes = TILE // per_byte
        tok_per_word = 4 * per_byte                      # 8 (INT4) or 16 (INT2) tokens per word
        word, q = np.divmod(r, tok_per_word)
        byte_in_row = 4 * word + (q % 4)                 # token q of a word sits in byte q mod 4
        slot = q // 4                                    # ... in nibble / 2-bit field q div 4
        addr = tile_base[:, None] + ch[None, :] * row_bytes + byte_in_row[:, None]
        shift = (slot * bits)[:, None] + 0 * ch[None, :]
    else:
        row_bytes = d // per_byte
        addr = tile_base[:, None] + r[:, None] * row_bytes + ch[None, :] // per_byte
        shift = (ch[None, :] % per_byte) * bits + 0 * r[:, None]
    return addr, shift


def _write_codes(buf, addr, shift, codes, bits):
    """Clear then set the code bits (codes of other tokens sharing a byte are kept)."""
    mask = (1 << bits) - 1
    a = addr.ravel()
    s = shift.ravel().astype(np.uint8)
    np.bitwise_and.at(buf, a, (~(np.uint8(mask) << s)).astype(np.uint8))
    np.bitwise_or.at(buf, a, ((codes.ravel().astype(np.uint8) & mask) << s).astype(np.uint8))


def _read_codes(buf, addr, shift, bits):
    mask = (1 << bits) - 1
    return (buf[addr] >> shift.astype(np.uint8)) & mask


def _meta_addresses(geom: Geometry, plane_base: int, tile_bytes: int, codes_bytes: int, pos):
    t, r = np.divmod(pos, TILE)
    base = plane_base + t * tile_bytes + codes_bytes + r * geom.ng * 2     # [n]
    gi = np.arange(geom.ng)
    return base[:, None] + 2 * gi[None, :]                                  # scale at +0, offset at +1


def _c_addresses(geom: Geometry, plane_base: int, pos):
    t, r = np.divmod(pos, TILE)
    return plane_base + t * geom.r_tile + geom.r_codes + geom.meta + 2 * r


def pack_group(buf: np.ndarray, geom: Geometry, layer: int, group: int, comp: dict,
               start: np.ndarray, rows=None):
    """Write a compressed loop group into the cache bytes.

    comp: output of method.compress_group for x of shape [P, 2, B, H, n, d].
    start: int [B], first position written for each batch row.
    rows: the batch rows to write (default: all).
    """
    a_codes, a_s, a_o = comp["anchor"]           # [2, B, H, n, d], [2, B, H, n, ng] x2
    _, B, H, n, d = a_codes.shape
    P = geom.loops_per_group
    for kv in range(2):
        for b in (range(B) if rows is None else rows):
            pos = int(start[b]) + np.arange(n, dtype=np.int64)
            if n and pos[-1] >= geom.max_seq_len:
                raise ValueError("append past max_seq_len")
            for h in range(H):
                base = geom.region_offset(layer, group, b, h)
                pa = base + geom.anchor_plane(kv)
                addr, sh = _code_addresses(geom, pa, geom.a_tile, pos, 4, channel_major=(kv == 1))
                _write_codes(buf, addr, sh, a_codes[kv, b, h], 4)
                ma = _meta_addresses(geom, pa, geom.a_tile, geom.a_codes, pos)
                buf[ma] = a_s[kv, b, h]
                buf[ma + 1] = a_o[kv, b, h]
                for j in range(P - 1):
                    r_codes, r_s, r_o, c_bits = comp["res"][j]
                    pr = base + geom.res_plane(j, kv)
                    addr, sh = _code_addresses(geom, pr, geom.r_tile, pos, 2, channel_major=(kv == 1))
                    _write_codes(buf, addr, sh, r_codes[kv, b, h], 2)
                    mr = _meta_addresses(geom, pr, geom.r_tile, geom.r_codes, pos)
                    buf[mr] = r_s[kv, b, h]
                    buf[mr + 1] = r_o[kv, b, h]
                    ca = _c_addresses(geom, pr, pos)
                    cb = c_bits[kv, b, h].astype(np.uint16)
                    buf[ca] = (cb & 0xFF).astype(np.uint8)
                    buf[ca + 1] = (cb >> 8).astype(np.uint8)


def read_plane_tokens(buf: np.ndarray, geom: Geometry, layer: int, group: int, b: int, h: int,
                      kv: int, plane: str, j: int, n: int):
    """Read back positions 0..n-1 of one plane.

    plane 'anchor' -> (codes [n, d], scale bytes [n, ng], offset bytes [n, ng])
    plane 'res'    -> (codes, scale bytes, offset bytes, c bf16 bits [n])"""
    pos = np.arange(n, dtype=np.int64)
    base = geom.region_offset(layer, group, b, h)
    if plane == "anchor":
        pa = base + geom.anchor_plane(kv)
        addr, sh = _code_addresses(geom, pa, geom.a_tile, pos, 4, channel_major=(kv == 1))
        ma = _meta_addresses(geom, pa, geom.a_tile, geom.a_codes, pos)
        return _read_codes(buf, addr, sh, 4), buf[ma], buf[ma + 1]
    pr = base + geom.res_plane(j, kv)
    addr, sh = _code_addresses(geom, pr, geom.r_tile, pos, 2, channel_major=(kv == 1))
    mr = _meta_addresses(geom, pr, geom.r_tile, geom.r_codes, pos)
    ca = _c_addresses(geom, pr, pos)
    c_bits = buf[ca].astype(np.uint16) | (buf[ca + 1].astype(np.uint16) << 8)
    return _read_codes(buf, addr, sh, 2), buf[mr], buf[mr + 1], c_bits


def bits_per_element(head_dim: int, group_size: int, loops: int) -> dict:
    """Storage per element position over `loops` loops, in bits, from the record sizes.

    Anchor: 4-bit code + (scale, offset) bytes per group.  Each earlier loop:
    2-bit code + (scale, offset) bytes per group + one BF16 coefficient per
    vector.  BF16 baseline: 16 bits per loop ([EXPL] worked storage example)."""
    ng = head_dim // group_size
    anchor = 8.0 * (head_dim / 2 + 2 * ng) / head_dim
    resid = 8.0 * (head_dim / 4 + 2 * ng + 2) / head_dim
    total = anchor + (loops - 1) * resid
    bf16 = 16.0 * loops
    return {"anchor": anchor, "residual": resid, "total": total, "bf16": bf16,
            "reduction": 1.0 - total / bf16, "ratio": bf16 / total,
            "codes_only_ratio": bf16 / (4.0 + 2.0 * (loops - 1))}

"""CPU oracle for ResidualQuant KV compression and decode attention.

TEST INFRASTRUCTURE ONLY.  This package is plain float64 NumPy written from
the ResidualQuant pages; it exists to check the CUDA library.  Only the test
suite, __graft_entry__.smoke() and bench.py's CPU-baseline leg import it.
The product path (decode_attention_rq_gb300 and its CUDA library) never
imports, links or runs anything here, and nothing here imports the product.

What each module follows:
  formats.py  E4M3 and BF16 round-to-nearest-even, from the format definitions.
  method.py   group quantizer, least-squares coefficient, rotated residual,
              shared/chained reconstruction, single-query softmax attention.
  layout.py   the cache's byte layout (this library's format).
  this file   cache-level steps: compress and pack a loop group, rebuild a
              loop's K/V from the cache bytes, and decode attention over the
              cache plus the current token held in BF16.
"""
from __future__ import annotations

import numpy as np

from . import formats, method, layout
from .formats import (e4m3_encode, e4m3_decode, e4m3_round, bf16_encode, bf16_decode, bf16_round)
from .method import quantize, dequantize, ls_coefficient, compress_group, attention, hadamard_matrix
from .layout import Geometry, TILE, pack_group, read_plane_tokens, bits_per_element, paged_pool

__all__ = ["formats", "method", "layout", "Geometry", "TILE", "quantize", "dequantize",
           "ls_coefficient", "compress_group", "attention", "hadamard_matrix", "pack_group", "read_plane_tokens",
           "bits_per_element", "paged_pool", "append", "reconstruct", "decode_attention", "decode_attention_append",
           "e4m3_encode", "e4m3_decode", "e4m3_round", "bf16_encode", "bf16_decode", "bf16_round"]


def append(buf: np.ndarray, geom: Geometry, R: np.ndarray, layer: int, group: int,
           kv: np.ndarray, start, chained: bool = False, precision: str = "f32",
           scaling: str = "ls", rows=None, rotation: str = "dense") -> dict:
    """Compress the P loops of n new tokens and write them at positions start[b].. .

    kv: float64 [P, 2, B, H, n, d] (exact BF16 values), anchor = last loop.
    rows: the batch rows to write (default: all).
    Returns the compress_group result (codes, metadata, reconstructions)."""
    comp = compress_group(kv, R, geom.group_size, chained=chained, precision=precision, scaling=scaling,
                          rotation=rotation)
    pack_group(buf, geom, layer, group, comp, np.asarray(start, dtype=np.int64), rows=rows)
    return comp


def reconstruct(buf: np.ndarray, geom: Geometry, R: np.ndarray, layer: int, group: int,
                b: int, h: int, loop: int, n: int, chained: bool = False):
    """Decoder's view of loop `loop` (0-based; P-1 is the anchor) for positions 0..n-1.

    Shared anchor ([EXPL], shared-master paragraph): K_l = c_l * a_hat + R^T r_hat_l,
    two planes read.  Chained: K_l = c_l * K_{l+1} + R^T r_hat_l down from the
    anchor, reading every residual plane between l and the anchor.
    Returns (K_hat [n, d], V_hat [n, d]) float64."""
    P, g = geom.loops_per_group, geom.group_size
    out = []
    for kv in range(2):
        codes, s_b, o_b = read_plane_tokens(buf, geom, layer, group, b, h, kv, "anchor", 0, n)
        x = dequantize(codes, s_b, o_b, g)
        if loop < P - 1:
            # shared: one residual plane against the anchor; chained: every
            # plane from the anchor's neighbour down to this loop
            js = range(P - 2, loop - 1, -1) if chained else [loop]
            for j in js:
                rc, rs, ro, cbits = read_plane_tokens(buf, geom, layer, group, b, h, kv, "res", j, n)
                r_hat = dequantize(rc, rs, ro, g)
                x = bf16_decode(cbits)[:, None] * x + r_hat @ R
        out.append(x)
    return out[0], out[1]


def decode_attention(buf: np.ndarray, geom: Geometry, R: np.ndarray, layer: int, group: int,
                     loop: int, q: np.ndarray, k_cur: np.ndarray, v_cur: np.ndarray,
                     seq_lens, scale: float, chained: bool = False,
                     rows=None) -> np.ndarray:
    """Attention of one (layer, group, loop) decode call.

    Keys/values: the seq_lens[b] cached tokens rebuilt for this loop, plus the
    current token's K/V straight from the BF16 temporary buffer ([EXPL]: the
    current token stays in BF16 until its last loop has run).
    q: float64 [B, Hq, d]; k_cur, v_cur: float64 [B, H, d] (H = the cache's KV
    heads).  Hq = H is multi-head attention, the pages' models; Hq a multiple
    of H is grouped-query attention (a reading: query head qh attends with KV
    head qh // (Hq / H), consecutive query heads sharing one).  rows: optional
    iterable of (b, qh) to evaluate (others left NaN).  Returns float64 [B, Hq, d]."""
    B, Hq, d = q.shape
    H = geom.num_heads
    if Hq % H:
        raise ValueError("query heads must be a multiple of the KV heads")
    qpk = Hq // H
    out = np.full((B, Hq, d), np.nan)
    todo = rows if rows is not None else [(b, qh) for b in range(B) for qh in range(Hq)]
    for b, qh in todo:
        h = qh // qpk
        n = int(seq_lens[b])
        K, V = reconstruct(buf, geom, R, layer, group, b, h, loop, n, chained)
        K = np.concatenate([K, k_cur[b, h][None, :]], axis=0)
        V = np.concatenate([V, v_cur[b, h][None, :]], axis=0)
        out[b, qh] = attention(q[b, qh], K, V, scale)
    return out


def decode_attention_append(buf: np.ndarray, geom: Geometry, R: np.ndarray, layer: int, group: int,
                            q: np.ndarray, kv_cur: np.ndarray, seq_lens, scale: float,
                            chained: bool = False, scaling: str = "ls", precision: str = "f32",
                            rotation: str = "dense"):
    """The group's last-loop call followed by the current token's append.

    [EXPL], temporary-buffer paragraph: the loops of the current token stay in
    BF16 until the last loop (the anchor) has run; only then can the group be
    coded against its anchor.  So the anchor-loop call attends over the cache as
    it stands plus the BF16 token (decode_attention, loop P-1) and then the
    token of every loop is compressed into slot seq_lens[b] (append, one token).
    kv_cur: float64 [P, 2, B, H, d].  A row whose slot would pass the capacity
    is attended but not appended.  Returns (out [B, H, d], appended [B] bool)."""
    P = geom.loops_per_group
    seq = np.asarray(seq_lens, dtype=np.int64)
    out = decode_attention(buf, geom, R, layer, group, P - 1, q, kv_cur[P - 1, 0], kv_cur[P - 1, 1], seq, scale,
                           chained=chained)
    ok = (seq >= 0) & (seq + 1 <= geom.max_seq_len)
    rows = [int(b) for b in np.nonzero(ok)[0]]
    if rows:
        append(buf, geom, R, layer, group, kv_cur[:, :, :, :, None, :], np.where(ok, seq, 0),
               chained=chained, precision=precision, scaling=scaling, rows=rows, rotation=rotation)
    return out, ok


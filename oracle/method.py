"""ResidualQuant arithmetic, written out plainly in float64 (oracle).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py may import this package.  The product path
(the CUDA library and its Python binding) never does; the two share no code.

Sources, by page and section:
  [EXPL] "ResidualQuant stores looped-Transformer KV caches as 2-bit
         residuals" (learnaivisually.com explainer): the paragraph that
         defines the stored overlay (residual = KV(loop) - c x anchor, c a
         least-squares coefficient per key or value vector, a rotation
         applied before quantization, rebuild c x anchor + residual on
         chip); the paragraph on shared versus chained anchors and the
         BF16 temporary buffer; the worked storage example (INT4 anchor,
         INT2 residuals, FP8 scale and offset per channel group, one BF16
         coefficient per residual vector).
  [SUMM] ai4snews summary of the arXiv paper: overview (last-loop anchor,
         least-squares scaling, rotation of the residual rather than of the
         KV, per-loop INT4/INT2 mixed precision), the main-results paragraph
         (group size 32/16, effective bits count codes, FP8 scale and
         offset and the BF16 coefficient).

Readings of what the pages leave open:
  * group quantizer: asymmetric min/max.  offset o = E4M3(min), scale
    s = E4M3((max - min) / (2^b - 1)); both rounded BEFORE coding; codes are
    the nearest grid point o + k*s of the exact value (ties to even k),
    clamped to [0, 2^b - 1]; s == 0 gives all-zero codes.
  * c is computed against the dequantized anchor (the decoder only has it),
    is 0 when the reference vector is all zero, and is rounded to BF16
    before the residual is formed, so encoder and decoder agree.
  * R is applied as u = R (x - c_b * ref); reconstruction uses R^T.
  * chained variant: loop l is coded against the reconstruction of loop
    l+1, the last loop being the anchor.
  * precision of the residual and its rotation: the pages do not fix it.  The
    codes are decided by u, so the oracle takes u in the precision the device
    computes it: IEEE binary32, e = fma(-c_b, ref, x) rounded once, and each
    u_i = sum_k R[i,k] e_k as a chain of binary32 fused multiply-adds in
    channel order k = 0..d-1 (the plain definition of the sum).  In chained
    mode the encoder's reference for loop l-1 is rebuilt the same way
    (acc_i = sum_k R[k,i] r_hat_k in order, then fma(c_b, ref, acc)).
    precision="f64" keeps the float64 reading of the same formulas, used to
    bound the binary32 one.
  * Walsh-Hadamard rotation (rotation="hadamard", d a power of two): R =
    H_d / sqrt(d), H_d the Sylvester Hadamard matrix (entry (i, k) =
    (-1)^popcount(i & k)).  The explainer's related-explainers list points to a
    2-bit KV cache built on a Hadamard rotation, and the summary's ablation
    paragraph compares rotation methods with the rotation fixed offline; H_d /
    sqrt(d) is one fixed orthogonal R that needs no d x d product.  In
    binary32 it is taken as the fast transform computes it: butterfly stages
    h = 1, 2, 4, ..., d/2, each pair (j, j + h) with j & h == 0 becoming
    (a + b, a - b) rounded to binary32, then one binary32 product with the
    binary32 value of 1/sqrt(d).  R is symmetric, so R^T is the same transform.
"""
from __future__ import annotations

import numpy as np

from .formats import e4m3_round, e4m3_encode, e4m3_decode, bf16_round, bf16_encode, bf16_decode, fma_f32

__all__ = ["quantize", "dequantize", "ls_coefficient", "compress_group", "attention",
           "rotate_f32", "rotate_back_f32", "hadamard_matrix", "fwht_f32", "hadamard_f32",
           "ANCHOR_BITS", "RESIDUAL_BITS"]

ANCHOR_BITS = 4     # [EXPL] worked example; [SUMM] overview (INT4 anchor)
RESIDUAL_BITS = 2   # [EXPL] worked example; [SUMM] overview (INT2 residuals)


def _nearest_grid_codes(v: np.ndarray, o: np.ndarray, s: np.ndarray, qmax: int) -> np.ndarray:
    """k minimising |v - (o + k s)| over integers, ties to even k, then clamped to [0, qmax].

    For v given exactly (bf16 or fp32 values) and E4M3 o, s, the differences
    below are exact in float64, so this is the nearest point of the exact
    quotient, not of a rounded one.
    """
    t = v - o
    safe_s = np.where(s > 0, s, 1.0)
    k = np.rint(t / safe_s)
    r = t - k * safe_s
    k = k + (2.0 * r > safe_s) - (2.0 * r < -safe_s)      # one step toward the nearest
    r = t - k * safe_s
    tie = (2.0 * np.abs(r) == safe_s)
    k = np.where(tie & (np.mod(k, 2.0) != 0.0), k + np.sign(r), k)
    k = np.clip(k, 0, qmax)
    return np.where(s > 0, k, 0.0).astype(np.uint8)


def quantize(v: np.ndarray, bits: int, g: int):
    """Group quantizer.  v: float64 [..., d]; groups are consecutive runs of g channels.

    Returns (codes uint8 [..., d], scale E4M3 bytes [..., d/g], offset E4M3 bytes [..., d/g]).
    """
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    if d % g:
        raise ValueError("head_dim must be a multiple of the group size")
    qmax = (1 << bits) - 1
    vg = v.reshape(v.shape[:-1] + (d // g, g))
    lo = vg.min(axis=-1)
    hi = vg.max(axis=-1)
    o = e4m3_round(lo)
    s = e4m3_round((hi - lo) / qmax)
    codes = _nearest_grid_codes(vg, o[..., None], s[..., None], qmax)
    return codes.reshape(v.shape), e4m3_encode(s), e4m3_encode(o)


def dequantize(codes: np.ndarray, scale_b: np.ndarray, offset_b: np.ndarray, g: int) -> np.ndarray:
    """x_hat = s * code + o per group, float64 (exact)."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    s = e4m3_decode(scale_b)[..., None]
    o = e4m3_decode(offset_b)[..., None]
    cg = codes.reshape(codes.shape[:-1] + (d // g, g)).astype(np.float64)
    return (s * cg + o).reshape(codes.shape)


def ls_coefficient(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """c = <x, y> / <y, y> over the last axis, 0 where <y, y> == 0 ([EXPL]: a
    least-squares coefficient per key or value vector)."""
    num = np.sum(x * y, axis=-1)
    den = np.sum(y * y, axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)


def rotate_f32(R: np.ndarray, e: np.ndarray) -> np.ndarray:
    """u = R e per vector in binary32: u_i accumulates fma(R[i,k], e_k, u_i) for
    k = 0..d-1.  R [d, d] and e [..., d] hold binary32 values; returns float32."""
    R = np.asarray(R, dtype=np.float32)
    e = np.asarray(e, dtype=np.float32)
    u = np.zeros(e.shape, dtype=np.float32)
    for k in range(e.shape[-1]):
        u = fma_f32(R[:, k], e[..., k:k + 1], u)
    return u


def rotate_back_f32(R: np.ndarray, r: np.ndarray) -> np.ndarray:
    """acc = R^T r per vector in binary32: acc_i accumulates fma(R[k,i], r_k, acc_i)
    for k = 0..d-1; returns float32."""
    R = np.asarray(R, dtype=np.float32)
    r = np.asarray(r, dtype=np.float32)
    acc = np.zeros(r.shape, dtype=np.float32)
    for k in range(r.shape[-1]):
        acc = fma_f32(R[k, :], r[..., k:k + 1], acc)
    return acc


def hadamard_matrix(d: int) -> np.ndarray:
    """H_d / sqrt(d) in float64 (d a power of two), from the Sylvester recursion
    H_2n = [[H_n, H_n], [H_n, -H_n]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("the Walsh-Hadamard rotation needs d a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H / np.sqrt(d)


def fwht_f32(e: np.ndarray) -> np.ndarray:
    """Unnormalized fast Walsh-Hadamard transform over the last axis in binary32:
    for h = 1, 2, 4, ..., d/2 every pair (j, j + h) with j & h == 0 becomes
    (a + b, a - b), each sum rounded to binary32."""
    v = np.array(e, dtype=np.float32)
    d = v.shape[-1]
    lead = v.shape[:-1]
    h = 1
    while h < d:
        w = v.reshape(lead + (d // (2 * h), 2, h))
        a, b = w[..., 0, :], w[..., 1, :]
        v = np.stack([a + b, a - b], axis=-2).reshape(lead + (d,))
        h *= 2
    return v


def hadamard_f32(e: np.ndarray) -> np.ndarray:
    """u = H_d e / sqrt(d) in binary32: the butterflies, then one product with the
    binary32 value of 1/sqrt(d); returns float32."""
    d = np.asarray(e).shape[-1]
    return (fwht_f32(e) * np.float32(1.0 / np.sqrt(d))).astype(np.float32)


def norm_ratio_coefficient(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """c = ||x|| / ||y|| over the last axis, 0 where ||y|| == 0.  The scaling the
    arXiv summary lists beside least squares among the appendix comparisons
    (ablation paragraph); the pages give no formula, so this takes the plain
    ratio of L2 norms, computed as sqrt(sum x^2 / sum y^2)."""
    num = np.sum(x * x, axis=-1)
    den = np.sum(y * y, axis=-1)
    return np.where(den > 0, np.sqrt(num / np.where(den > 0, den, 1.0)), 0.0)


def compress_group(x: np.ndarray, R: np.ndarray, g: int, chained: bool = False, precision: str = "f32",
                   scaling: str = "ls", rotation: str = "dense"):
    """Compress the P loops of one loop group.

    x: float64 [P, ..., d], loop index first, the last loop is the anchor
       ([EXPL]: the final loop's KV is the INT4 master; [SUMM]: last-loop anchor).
    R: [d, d], the fixed rotation as the device receives it (binary32 values).
    precision: "f32" (the residual and rotation as the device computes them,
       see the module docstring) or "f64".
    scaling: "ls" (least-squares coefficient, the method's) or "norm" (norm ratio).
    rotation: "dense" (u = R e as given) or "hadamard" (R must then be
       hadamard_matrix(d); the binary32 path takes the fast transform).
    Returns a dict with
      anchor: (codes, scale_b, offset_b)
      res[j] for j in 0..P-2: (codes, scale_b, offset_b, c_bf16_bits)
      u[j]: the rotated residual before quantization (float64 array)
      recon: float64 [P, ..., d], the decoder's view of every loop, computed
             in float64 from the stored values (c_b * ref_hat + R^T r_hat)
    """
    x = np.asarray(x, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    P = x.shape[0]
    a_codes, a_s, a_o = quantize(x[P - 1], ANCHOR_BITS, g)
    a_hat = dequantize(a_codes, a_s, a_o, g)
    recon = np.empty_like(x)
    recon[P - 1] = a_hat
    res, us = [None] * (P - 1), [None] * (P - 1)
    enc_ref = a_hat                                   # the encoder's reference (chained: rebuilt loop)
    for j in range(P - 2, -1, -1):
        ref = enc_ref if chained else a_hat
        c = ls_coefficient(x[j], ref) if scaling == "ls" else norm_ratio_coefficient(x[j], ref)
        c_bits = bf16_encode(c)
        cb = bf16_decode(c_bits)[..., None]
        if precision == "f32":
            e = fma_f32(-cb, ref, x[j])               # residual, one binary32 rounding
            u = (hadamard_f32(e) if rotation == "hadamard" else rotate_f32(R, e)).astype(np.float64)
        else:
            e = x[j] - cb * ref
            u = e @ R.T
        r_codes, r_s, r_o = quantize(u, RESIDUAL_BITS, g)
        r_hat = dequantize(r_codes, r_s, r_o, g)
        dec_ref = recon[j + 1] if chained else a_hat
        recon[j] = cb * dec_ref + r_hat @ R           # R^T r_hat for each vector, float64
        if chained:
            if precision == "f32":
                back = hadamard_f32(r_hat) if rotation == "hadamard" else rotate_back_f32(R, r_hat)
                enc_ref = fma_f32(cb, enc_ref, back).astype(np.float64)
            else:
                enc_ref = recon[j]
        res[j] = (r_codes, r_s, r_o, c_bits)
        us[j] = u
    return {"anchor": (a_codes, a_s, a_o), "res": res, "u": us, "recon": recon}


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Single-query softmax attention, float64: softmax(scale * K q) V.

    q [d], K [n, d], V [n, d] -> [d].  The maximum is subtracted before exp."""
    s = scale * (K @ q)
    m = np.max(s)
    p = np.exp(s - m)
    return (p @ V) / np.sum(p)

// The current token's append, run by the merge CTAs of the anchor-loop call.
//
// Once the group's last loop has produced its K/V, every loop's current token
// is known and can join the compressed cache; until then it sits in the BF16
// temporary buffer (the explainer "ResidualQuant stores looped-Transformer KV
// caches as 2-bit residuals", paragraph on the temporary buffer, and the
// stored-overlay paragraph for what is stored).  The anchor-loop call does it
// in its merge kernel, one CTA per (row, head), K and V, all P loops, with the
// arithmetic of the append kernel (same quantizer decisions, same float32
// operation order), so the stored bytes equal those of rq_append with
// n_tokens = 1.  One CTA codes K, another V; thread = channel (128 threads).
//
// The CTA is small on purpose: 128 threads, at most 32 registers a thread and
// a few KB of shared memory fit on an SM beside the decode kernel's three
// CTAs, so the merge CTAs start at once (launched as programmatic dependents)
// and do the append's work while the decode kernel streams the cache.  Split
// around the grid-dependency wait:
//   * token_append_compute (before the wait): loads the token, quantizes the
//     anchor, takes the coefficients, rotates and quantizes the residuals, and
//     reads the channel-major V words it will rewrite.  It only reads the
//     cache, and only words the decode kernel also only reads.
//   * token_append_store (after the wait): writes the codes, metadata and
//     coefficients of the new slot.  After the wait no kernel of the stream
//     before this one is running, so no copy of the decode kernel can see a
//     half-written slot.
#pragma once

#include "rq_quant.cuh"

namespace rq {
namespace {

constexpr int kAppendThreads = 128;   // thread = channel (d <= 128)
constexpr int kRotChunk = 4;          // residual loops rotated per pass over R

// Dynamic shared memory of the append (one vector type, K or V), carved for P
// loops in 16-byte aligned pieces.
struct TokenAppendSmem {
  float* e;          // [kRotChunk][128] residuals of the loops in the current pass; then u
  float* ref;        // [128] dequantized anchor (shared) or rebuilt loop l+1 (chained)
  float* rhat;       // [128] chained: dequantized rotated residual of the current loop
  float* cb;         // [kMaxLoops] coefficient per residual loop (float)
  uint32_t* vword;   // [P][128] V: the channel-major code word of the new slot, per plane
  __nv_bfloat16* x;  // [P][128] the token of every loop (exact BF16 values)
  uint8_t* code;     // [P][128] codes per plane (plane P-1: the anchor)
  uint16_t* meta;    // [P][8] (scale, offset) bytes per plane and group
  uint16_t* cbits;   // [P] BF16 coefficient per residual plane

  __host__ __device__ static size_t bytes(int P) {
    return kRotChunk * 128 * 4 + 128 * 4 * 2 + kMaxLoops * 4 + (size_t)P * 128 * 4 + (size_t)P * 128 * 2 +
           (size_t)P * 128 + (size_t)P * 8 * 2 + ((size_t)P * 2 + 15) / 16 * 16;
  }
  __device__ TokenAppendSmem(uint8_t* base, int P) {
    e = reinterpret_cast<float*>(base);
    base += kRotChunk * 128 * 4;
    ref = reinterpret_cast<float*>(base);
    base += 128 * 4;
    rhat = reinterpret_cast<float*>(base);
    base += 128 * 4;
    cb = reinterpret_cast<float*>(base);
    base += kMaxLoops * 4;
    vword = reinterpret_cast<uint32_t*>(base);
    base += (size_t)P * 128 * 4;
    x = reinterpret_cast<__nv_bfloat16*>(base);
    base += (size_t)P * 128 * 2;
    code = base;
    base += (size_t)P * 128;
    meta = reinterpret_cast<uint16_t*>(base);
    base += (size_t)P * 8 * 2;
    cbits = reinterpret_cast<uint16_t*>(base);
  }
};

// Where the new slot's codes, metadata and coefficient go in one plane.
struct SlotRef {
  uint8_t* tile;      // start of the tile holding the slot
  int row;            // slot within the tile
  int bits, per_byte;
  int64_t codes_bytes;
};

// The slot of plane p (P-1: the anchor) of (layer, group, b, h); `page` is the
// slot's tile's page in the paged layout.
__device__ __forceinline__ SlotRef slot_in_plane(const Geom& g, uint8_t* base, int layer, int group, int b, int h,
                                                 int page, int p, int kvi, int pos) {
  const bool anchor = p == g.P - 1;
  SlotRef r;
  r.bits = anchor ? kAnchorBits : kResBits;
  r.per_byte = 8 / r.bits;
  r.codes_bytes = anchor ? g.a_codes : g.r_codes;
  r.tile = base + g.tile_offset(layer, group, b, h, anchor, p, kvi, pos / kTile, page);
  r.row = pos % kTile;
  return r;
}

// Channel-major V: the 32-bit word of channel i that holds the slot, and the
// bit position of the slot's field in it (slot q of a word: byte q % 4, field q / 4).
__device__ __forceinline__ uint32_t* vword_ptr(const SlotRef& r, int i, int* shift) {
  const int tpw = 4 * r.per_byte, q = r.row % tpw;
  *shift = 8 * (q & 3) + r.bits * (q >> 2);
  return reinterpret_cast<uint32_t*>(r.tile + i * (kTile / r.per_byte) + (r.row - q) / r.per_byte);
}

// 2-bit codes of this thread's element of the rotated residuals held in
// s.e[jj * 128 + i], loops j0 + jj (jj < nj).
__device__ __forceinline__ void quantize_residuals(const TokenAppendSmem& s, int nj, int j0, int gs, int i, bool act) {
#pragma unroll 1
  for (int jj = 0; jj < nj; ++jj) {
    uint8_t sb, ob;
    float vh;
    const int code = quantize_lane(s.e[jj * 128 + i], act, gs, 3, &sb, &ob, &vh);
    const int j = j0 + jj;
    s.code[j * 128 + i] = (uint8_t)code;
    if (act && i % gs == 0) s.meta[j * 8 + i / gs] = (uint16_t)sb | ((uint16_t)ob << 8);
    s.rhat[i] = act ? vh : 0.f;   // chained mode rebuilds from it (nj = 1 there)
  }
}

// u_t[i] = sum_k R[i][k] e_t[k] for the NJ residuals in s.e, k ascending, one
// float32 FMA chain each (the append kernel's order), or the fast Walsh-Hadamard
// transform (RQ_MODE_HADAMARD); then u replaces e.
template <int D, int NJ>
__device__ __forceinline__ void rotate_chunk(const TokenAppendSmem& s, const float4* Rrow, int i, bool act,
                                             bool hadamard) {
  float u[NJ];
  if (hadamard) {   // d = 128; s.e serves as the butterflies' scratch (each thread reads its own slot first)
#pragma unroll
    for (int t = 0; t < NJ; ++t) u[t] = s.e[t * 128 + i];
    hadamard128<NJ>(u, i, s.e);
    __syncthreads();
#pragma unroll
    for (int t = 0; t < NJ; ++t) s.e[t * 128 + i] = u[t];
    return;
  }
#pragma unroll
  for (int t = 0; t < NJ; ++t) u[t] = 0.f;
#pragma unroll 8
  for (int k4 = 0; k4 < D / 4; ++k4) {
    const float4 r = __ldg(Rrow + k4);
#pragma unroll
    for (int t = 0; t < NJ; ++t) {
      const float4 x = *reinterpret_cast<const float4*>(s.e + t * 128 + 4 * k4);
      u[t] = fmaf(r.x, x.x, u[t]);
      u[t] = fmaf(r.y, x.y, u[t]);
      u[t] = fmaf(r.z, x.z, u[t]);
      u[t] = fmaf(r.w, x.w, u[t]);
    }
  }
  __syncthreads();   // every thread has read the residuals: u takes their place
#pragma unroll
  for (int t = 0; t < NJ; ++t) s.e[t * 128 + i] = act ? u[t] : 0.f;
}

// Before the wait: the append of vector type kvi (0 = K, 1 = V).  Returns
// whether the slot fits (same on every thread); a row whose slot would
// overflow the capacity is skipped and status[1] set, one whose page entry is
// out of range is skipped and status[2] set.  *page: the slot's page (paged layout).
template <int D>
__device__ bool token_append_compute(const Geom& g, uint8_t* base, const float* R, const __nv_bfloat16* kv,
                                     int batch, int layer, int group, int b, int h, int kvi, int pos,
                                     int32_t* status, uint8_t* smem, int* page) {
  const int P = g.P, gs = g.g;
  const TokenAppendSmem s(smem, P);
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const bool act = i < D;
  const bool chained = (g.mode & RQ_MODE_CHAINED) != 0;
  const bool norm_ratio = (g.mode & RQ_MODE_NORM_RATIO) != 0;
  const bool hadamard = (g.mode & RQ_MODE_HADAMARD) != 0;
  if (pos < 0 || pos + 1 > g.Nmax) {
    if (i == 0 && status) atomicExch(&status[1], 1);
    return false;
  }
  *page = 0;
  if (g.paged) {
    *page = checked_page(g, raw_page(g, b, pos / kTile), status);
    if (*page < 0) return false;
  }
#pragma unroll 4
  for (int l = 0; l < P; ++l)   // block (l, kvi) of the temporary buffer
    s.x[l * 128 + i] = act ? kv[((((size_t)l * 2 + kvi) * batch + b) * g.H + h) * D + i] : __float2bfloat16(0.f);
  if (act && kvi == 1) {
#pragma unroll 4
    for (int l = 0; l < P; ++l) {
      int sh;
      s.vword[l * 128 + i] = *vword_ptr(slot_in_plane(g, base, layer, group, b, h, *page, l, 1, pos), i, &sh);
    }
  }
  __syncthreads();

  // anchor: loop P-1, 4-bit codes
  {
    uint8_t sb, ob;
    float vh;
    const int code = quantize_lane(__bfloat162float(s.x[(P - 1) * 128 + i]), act, gs, 15, &sb, &ob, &vh);
    s.code[(P - 1) * 128 + i] = (uint8_t)code;
    s.ref[i] = act ? vh : 0.f;
    if (act && i % gs == 0) s.meta[(P - 1) * 8 + i / gs] = (uint16_t)sb | ((uint16_t)ob << 8);
  }
  __syncthreads();

  const float4* Rrow = hadamard ? nullptr : reinterpret_cast<const float4*>(R + (size_t)(act ? i : 0) * D);
  if (!chained) {
    // coefficients of every residual loop against the anchor, one warp each
#pragma unroll 1
    for (int j = warp; j < P - 1; j += kAppendThreads / 32) {
      const uint16_t bits = coefficient_bits(s.x + j * 128, s.ref, D, norm_ratio, lane);
      if (lane == 0) {
        s.cbits[j] = bits;
        s.cb[j] = bf16_bits_to_f32(bits);
      }
    }
    __syncthreads();
    // residuals of up to kRotChunk loops, one pass over row i of R for all of them
#pragma unroll 1
    for (int j0 = 0; j0 < P - 1; j0 += kRotChunk) {
      const int nj = min(kRotChunk, P - 1 - j0);
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj)
        s.e[jj * 128 + i] = fmaf(-s.cb[j0 + jj], s.ref[i], __bfloat162float(s.x[(j0 + jj) * 128 + i]));
      __syncthreads();
      switch (nj) {
        case 1: rotate_chunk<D, 1>(s, Rrow, i, act, hadamard); break;
        case 2: rotate_chunk<D, 2>(s, Rrow, i, act, hadamard); break;
        case 3: rotate_chunk<D, 3>(s, Rrow, i, act, hadamard); break;
        default: rotate_chunk<D, 4>(s, Rrow, i, act, hadamard); break;
      }
      quantize_residuals(s, nj, j0, gs, i, act);
      __syncthreads();
    }
  } else {
    // chained: loop j against the rebuilt loop j+1, from P-2 down
#pragma unroll 1
    for (int j = P - 2; j >= 0; --j) {
      if (warp == 0) {
        const uint16_t bits = coefficient_bits(s.x + j * 128, s.ref, D, norm_ratio, lane);
        if (lane == 0) {
          s.cbits[j] = bits;
          s.cb[j] = bf16_bits_to_f32(bits);
        }
      }
      __syncthreads();
      s.e[i] = act ? fmaf(-s.cb[j], s.ref[i], __bfloat162float(s.x[j * 128 + i])) : 0.f;
      __syncthreads();
      rotate_chunk<D, 1>(s, Rrow, i, act, hadamard);
      quantize_residuals(s, 1, j, gs, i, act);
      if (j > 0) {
        // rebuilt loop j = cb * ref + R^T r_hat becomes the reference of loop j-1
        __syncthreads();
        float acc = 0.f;
        if (hadamard) {   // R^T = R; s.e is free here
          float v[1] = {s.rhat[i]};
          hadamard128<1>(v, i, s.e);
          acc = v[0];
        } else if (act) {
#pragma unroll 8
          for (int k = 0; k < D; ++k) acc = fmaf(__ldg(R + (size_t)k * D + i), s.rhat[k], acc);
        }
        __syncthreads();
        if (act) s.ref[i] = fmaf(s.cb[j], s.ref[i], acc);
      }
      __syncthreads();
    }
  }
  return true;
}

// After the wait: the new slot's bytes of vector type kvi in every plane (call
// only when token_append_compute returned true).
template <int D>
__device__ void token_append_store(const Geom& g, uint8_t* base, int layer, int group, int b, int h, int kvi,
                                   int pos, int page, uint8_t* smem) {
  const int P = g.P, gs = g.g;
  const TokenAppendSmem s(smem, P);
  const int i = threadIdx.x;
  const bool act = i < D;
#pragma unroll 1
  for (int p = 0; p < P; ++p) {
    const SlotRef r = slot_in_plane(g, base, layer, group, b, h, page, p, kvi, pos);
    if (kvi == 0) {
      // K rows are token-major: byte m of the slot's row holds channels m*per_byte ..
      const int row_bytes = D / r.per_byte;
      if (i < row_bytes) {
        uint32_t byte = 0;
        for (int m = 0; m < r.per_byte; ++m) byte |= (uint32_t)s.code[p * 128 + i * r.per_byte + m] << (r.bits * m);
        r.tile[r.row * row_bytes + i] = (uint8_t)byte;
      }
    } else if (act) {
      // V rows are channel-major: this channel's word, the slot's field replaced
      int sh;
      uint32_t* wp = vword_ptr(r, i, &sh);
      const uint32_t fmask = (1u << r.bits) - 1u;
      *wp = (s.vword[p * 128 + i] & ~(fmask << sh)) | ((uint32_t)s.code[p * 128 + i] << sh);
    }
    if (act && i % gs == 0)
      *reinterpret_cast<uint16_t*>(r.tile + r.codes_bytes + r.row * g.ng * 2 + (i / gs) * 2) = s.meta[p * 8 + i / gs];
    if (p < P - 1 && i == 0)
      *reinterpret_cast<uint16_t*>(r.tile + r.codes_bytes + g.meta + r.row * 2) = s.cbits[p];
  }
}

}  // namespace
}  // namespace rq

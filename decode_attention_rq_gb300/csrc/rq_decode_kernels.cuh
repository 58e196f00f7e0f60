// The decode path's kernels (query prep, the streaming decode kernel, the
// merge) and their launcher, shared by rq_decode.cu (calls reading up to three
// residual planes) and rq_decode_chained.cu (chained calls reading four to
// seven, instantiated in their own translation unit so the two compile in
// parallel).  The design notes are at the top of rq_decode.cu.
#pragma once

#include <atomic>

#include <cuda_fp8.h>
#include "rq_internal.cuh"
#include "rq_token_append.cuh"

namespace rq {

struct DecodeArgs {
  Geom g;
  const uint8_t* base;
  const float* R;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cur;
  const __nv_bfloat16* v_cur;
  const int32_t* seq_lens;
  float* out;
  int32_t* status;
  const __nv_bfloat16* kv_all;   // [P][2][batch][H][d]: the anchor-loop call also appends it; else NULL
  float* partials;       // [(C + batch*H)][pstride]: (m, l, acc_anchor[d], acc_residual[d])
  uint32_t* packs;       // [batch*H][kPackWords]: query operands of the scoring products
  int pstride;
  int layer, group, batch, res0;   // res0: first residual plane this loop reads
  int qh;                          // query heads a work unit covers (1; grouped-query: 2 or 4)
  float qscale;                    // softmax_scale * log2(e)
};

// Chained calls that read 4 to 7 residual planes (rq_decode_chained.cu).
cudaError_t launch_decode_long_chain(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream);
// Grouped-query calls reading at most one residual plane, a.qh (2 or 4) query
// heads per work unit (rq_decode_gqa.cu).
cudaError_t launch_decode_gqa(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream);

// Query operands per (row, query head): a header (two scales, the per-group sums
// of the query and of the rotated query) then the f16 B-operand images of the
// scoring products, 8 lanes x (anchor + residual) registers.
constexpr int kPackHeader = 32;
constexpr int kPackWords = kPackHeader + 8 * 32;

namespace {

constexpr int kThreads = 256;
constexpr int kMaxCtasPerSm = 3;     // the workspace holds partials for this many CTAs per SM
constexpr int kMaxRows = RQ_MAX_DECODE_BATCH;   // batch rows one call may cover
constexpr int kMaxRes = 7;             // residual planes one call may read (chained, 8 loops)
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPrepThreads = 256;
constexpr int kMergeThreads = 256;
constexpr int kMaxContrib = 512;       // decode CTAs one merge can combine (the grid is smaller)
// Value-weight image of one (plane, group): per value product m (8) and lane t
// (4) the B registers b0, b1 (8 B), hi pieces at +0 and lo pieces at +kWPiece.
// The strides put the pieces 8 banks apart and neighbouring images 2 banks
// apart, so the lanes' stores and loads do not collide in shared memory.
constexpr int kWPiece = 288;
constexpr int kWItem = 648;

__device__ __forceinline__ float2 meta2(const uint8_t* p) {   // (scale, offset)
  return e4m3x2_to_f32x2(*reinterpret_cast<const uint16_t*>(p));
}
__device__ __forceinline__ int clamp_len(int n, int nmax) { return n < 0 ? 0 : (n > nmax ? nmax : n); }

// ---- f16 tensor-core products ------------------------------------------------
// d += a b for one 16 x 8 x 16 tile: A 16 x 16 row-major f16, B 16 x 8 f16, D f32.
// Fragments (lane = 4 g + t): a0 (row g, k 2t, 2t+1), a1 (row g+8, same k),
// a2 (row g, k 2t+8, 2t+9), a3 (row g+8, those k); b0 (k 2t, 2t+1; col g),
// b1 (k 2t+8, 2t+9; col g); d0 (row g, col 2t), d1 (row g, col 2t+1), d2, d3
// (row g+8, cols 2t, 2t+1).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Codes as f16 operands.  An f16 whose bit pattern is an integer n < 2048 has the
// value n * 2^-24 (subnormals, then the first normal binade, share the step
// 2^-24), so masking a code word leaves exact f16 multiples of the codes: no
// conversion and no bias.  The tensor core keeps such operands exactly.
//
// INT4 word (byte i = element 2i in bits 0-3, element 2i+1 in bits 4-7): four
// f16x2 registers, r[k] half h = element k + 4h; odd k carry 16 x the code.
__device__ __forceinline__ void int4_f16(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t w8 = w >> 8;
  r[0] = w & 0x000F000Fu;
  r[1] = w & 0x00F000F0u;
  r[2] = w8 & 0x000F000Fu;
  r[3] = w8 & 0x00F000F0u;
}
// INT2 word (byte i, bits 2m..2m+1 = element 4i + m): eight f16x2 registers,
// r[2m + hb] half h = element 4 (hb + 2h) + m, carrying 4^m x the code.
__device__ __forceinline__ void int2_f16(uint32_t w, uint32_t (&r)[8]) {
  const uint32_t w8 = w >> 8;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    r[2 * m] = w & (0x00030003u << (2 * m));
    r[2 * m + 1] = w8 & (0x00030003u << (2 * m));
  }
}
__device__ __forceinline__ uint32_t pack_f16x2(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}
// x as two f16 pieces hi + lo (about 22 significant bits; magnitudes past the
// f16 range clamp to +-65504)
__device__ __forceinline__ void f16_pieces(float x, __half& hi, __half& lo) {
  x = fminf(fmaxf(x, -65504.f), 65504.f);
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
}
// (x0, x1) rounded to f16, saturating at +-65504: x0 in the low half
__device__ __forceinline__ uint32_t f16x2_sat(float x0, float x1) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x1), "f"(x0));
  return r;
}
// f16x2 pieces of (x0, x1): hi = the rounded pair, lo = the rounded remainders
__device__ __forceinline__ void f16x2_pieces(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = f16x2_sat(x0, x1);
  const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  lo = f16x2_sat(x0 - h.x, x1 - h.y);
}

// Balanced split of U units over C CTAs: CTA c takes [start(c), start(c+1)) with
// start(c) = c*q + min(c, rem), q = U / C, rem = U % C (32-bit arithmetic only).
struct Split {
  int q, rem;
  __device__ __forceinline__ int start(int c) const { return c * q + min(c, rem); }
  // CTA owning unit u (u < U)
  __device__ __forceinline__ int owner(int u) const {
    const int big = (q + 1) * rem;            // units held by the first rem CTAs
    return u < big ? u / (q + 1) : rem + (u - big) / q;
  }
};

template <int D, int GS, int NRES>
struct Cfg {
  static constexpr int NG = D / GS;
  static constexpr int A_CODES = kTile * D / 2;
  static constexpr int R_CODES = kTile * D / 4;
  static constexpr int META = kTile * NG * 2;
  static constexpr int A_TILE = A_CODES + META;
  static constexpr int R_TILE = R_CODES + META + kTile * 2;
  static constexpr int SUB = 2 * A_TILE + 2 * NRES * R_TILE;      // one 64-token layout tile
  static constexpr int UT = 2;                                    // layout tiles per work unit
  static constexpr int UTOK = UT * kTile;                         // tokens per work unit
  static constexpr int STAGE = UT * SUB;
  // Stage layout.  Contiguous cache: each plane's UT tiles together (K anchor,
  // V anchor, then K and V of each residual plane; PA, PR bytes per plane), as
  // a unit's tiles of a plane are neighbours in the cache: one copy per plane.
  // Paged cache: tile by tile (SUB bytes), each tile's anchor pair and its
  // residual planes being neighbours in the tile's page: two copies per tile.
  static constexpr int PA = UT * A_TILE;
  static constexpr int PR = UT * R_TILE;
  template <bool PAGED> struct Lay {
    static constexpr int TA = PAGED ? SUB : A_TILE;          // tile stride, anchor planes
    static constexpr int AV = PAGED ? A_TILE : PA;           // V anchor of tile 0
    static constexpr int RB = PAGED ? 2 * A_TILE : 2 * PA;   // K of residual plane 0, tile 0
    static constexpr int TR = PAGED ? SUB : R_TILE;          // tile stride, residual planes
    static constexpr int PL = PAGED ? R_TILE : PR;           // K to V, and plane to plane: 2 PL
  };
  // CTAs per SM: two while the registers allow; one from four residual planes up
  static constexpr int MINB = NRES <= 1 ? 3 : (NRES <= 3 ? 2 : 1);
  static constexpr int NITEM = NG * (1 + NRES);  // (plane, group) value-weight images
  static constexpr int WIMG = NITEM * kWItem + 256;              // + a zero block for idle lanes
  static constexpr int STAGES = (MINB * (3 * STAGE + WIMG) + MINB * 8192 <= 224 * 1024) ? 3 : 2;
  static constexpr int SMEM = STAGES * STAGE + WIMG;
  // CTAs per SM that the shared memory allows (MINB, or one fewer when MINB
  // copies of SMEM and the static part do not fit)
  static constexpr int FIT = (MINB * (SMEM + 8192) <= 228 * 1024 || MINB == 1) ? MINB : MINB - 1;
  // registers a thread: the share of FIT CTAs (a multiple of 8, at most 255); anchor-only
  // calls 72, leaving room for a token-append CTA of the merge kernel beside three CTAs
  static constexpr int MAXREG = NRES == 0 ? 72 : (65536 / (256 * FIT) / 8 * 8 > 255 ? 255 : 65536 / (256 * FIT) / 8 * 8);
  // ---- scoring products (tokens x channels), per warp 16 tokens ----
  // anchor K: lane t holds words [t WA, (t+1) WA) of a token row (8 channels each);
  // product j takes registers 2j, 2j+1 of the lane (word j/2)
  static constexpr int WA = D / 32;
  static constexpr int NMA = 2 * WA;
  // residual K: lanes t < TR hold words 2t, 2t+1 (16 channels each); product j
  // takes registers 2j, 2j+1 (word j/4)
  static constexpr int TR = D / 32;
  static constexpr int NMR = 8;
  static constexpr int NIMG = 2 * NMA + (NRES > 0 ? 2 * NMR : 0);   // B-operand registers per lane
  static_assert(kPackHeader + 8 * NIMG <= kPackWords, "query pack");
  // channel group of the anchor / residual product j for lane t
  static constexpr int ga(int t, int j) { return (t * WA + j / 2) * 8 / GS; }
  static constexpr int gr(int t, int j) { return (2 * t + j / 4) * 16 / GS; }
  // Products whose lanes all see the same groups share an accumulator: each
  // lane's channels land in its own column pair, so an accumulator holds, per
  // lane, the partial dot product of one group.  own: bit 4 a + t set when
  // (accumulator a, lane t) is the first to hold its group (it adds the group's
  // offset term).
  struct AccMap {
    int acc[8];   // accumulator of product j
    int rep[8];   // a product of accumulator a
    int n;        // accumulators
    unsigned own;
  };
  static constexpr AccMap make_map(bool res) {
    AccMap m{};
    const int nj = res ? NMR : NMA, nt = res ? TR : 4;
    for (int j = 0; j < nj; ++j) {
      int found = -1;
      for (int a = 0; a < m.n && found < 0; ++a) {
        bool same = true;
        for (int t = 0; t < nt; ++t)
          if ((res ? gr(t, j) : ga(t, j)) != (res ? gr(t, m.rep[a]) : ga(t, m.rep[a]))) same = false;
        if (same) found = a;
      }
      if (found < 0) {
        found = m.n;
        m.rep[m.n++] = j;
      }
      m.acc[j] = found;
    }
    for (int a = 0; a < m.n; ++a)
      for (int t = 0; t < nt; ++t) {
        const int g = res ? gr(t, m.rep[a]) : ga(t, m.rep[a]);
        bool first = true;
        for (int a2 = 0; a2 <= a; ++a2)
          for (int t2 = 0; t2 < nt; ++t2) {
            if (a2 == a && t2 >= t) continue;
            if ((res ? gr(t2, m.rep[a2]) : ga(t2, m.rep[a2])) == g) first = false;
          }
        if (first) m.own |= 1u << (4 * a + t);
      }
    return m;
  }
  static constexpr int NACA = make_map(false).n;
  static constexpr int NACR = make_map(true).n;
  // ---- value products (channels x tokens), per warp 16 channels ----
  static constexpr int VW = D / 16;   // warps with a 16-channel tile
  static constexpr int NGW = (NG + 3) / 4;   // weight groups per lane: t, t + 4
};

// Byte offset of token t's slot in a value-weight image (within a piece), and
// the power of two the weight is scaled by so that it cancels the code's own
// factor (16 for the high nibbles of INT4 words, 4^m for field m of INT2 words).
// In both layouts an f16x2 operand holds tokens t and t + 2 (t mod 4 < 2): the
// pair shares one 4-byte slot, low half first, and one factor.
__device__ __forceinline__ void int4_slot(int tok, int& off, float& sc) {
  const int tau = tok >> 6, tp = tok & 63, w = tp >> 3, i = tp & 7;
  const int lane = w >> 1, e = w & 1;
  const int k = 2 * (i & 1) + ((i >> 2) & 1), h = (i >> 1) & 1;
  const int rho = 4 * (2 * tau + e) + k;
  off = ((rho >> 1) * 4 + lane) * 8 + (rho & 1) * 4 + h * 2;
  sc = (k & 1) ? 0.0625f : 1.f;
}
__device__ __forceinline__ void int2_slot(int tok, int& off, float& sc) {
  const int tau = tok >> 6, tp = tok & 63, lane = tp >> 4, q = tp & 15;
  const int m = q >> 2, i = q & 3, hb = i & 1, h = i >> 1;
  const int rho = 8 * tau + 2 * m + hb;
  off = ((rho >> 1) * 4 + lane) * 8 + (rho & 1) * 4 + h * 2;
  sc = m == 0 ? 1.f : (m == 1 ? 0.25f : (m == 2 ? 0.0625f : 0.015625f));
}

// Query prep: one CTA per (row, query head).  Applies R to the query and writes
// the B operands of the scoring products: for q (anchor plane) and R q (residual
// planes), a power-of-two scale 2^k bringing max |x| into [2^14, 2^15), each
// channel as two f16 pieces of x 2^k (divided by the code factor of its slot),
// placed in the register order of the lane that holds the matching codes.
template <int D, int GS, int NRES>
__global__ void __launch_bounds__(kPrepThreads) qprep_kernel(DecodeArgs a) {
  using C = Cfg<D, GS, NRES>;
  constexpr int NG = C::NG, NMA = C::NMA, NIMG = C::NIMG;
  constexpr int RPW = 16;                  // rows of R per warp (D / 8 <= 16; the rest padded)
  __shared__ __align__(16) float q_s[D];
  __shared__ float qr_s[D];
  __shared__ float red_s[2][kPrepThreads / 32];
  __shared__ __align__(16) uint32_t pack_s[kPackWords];
  const int bh = blockIdx.x, tid = threadIdx.x;
  // R first (R stays unchanged while the cache is used), before waiting for the
  // kernel ahead of this one.  Warp w holds rows w, w+8, ...; lane l columns
  // 4l..4l+3, so each warp-wide load reads one contiguous row.
  const int lane = tid & 31, warp = tid >> 5;
  const bool hadamard = (a.g.mode & RQ_MODE_HADAMARD) != 0;   // fast transform instead of R (d = 128)
  float4 rv[NRES > 0 ? RPW : 1];
  if (NRES > 0 && !hadamard) {
#pragma unroll
    for (int v = 0; v < RPW; ++v) {
      const int row = warp + 8 * v;
      rv[v] = (row < D && lane < D / 4) ? __ldg(reinterpret_cast<const float4*>(a.R + (size_t)row * D) + lane)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // Launched as a programmatic dependent of whatever precedes the call on the
  // stream.  The query and R are inputs, complete before that work releases
  // this kernel (the contract in rq.h), so the whole pack is built before the
  // wait, while the previous call drains; only its write to the workspace
  // (which the previous call's decode kernel may still read) waits.  The
  // decode kernel is released at once: it splits the work and starts its
  // first cache copies.  What it reads before its own wait (seq_lens, the
  // cache) no kernel of this library writes while released early: the kernels
  // that write the cache (the append kernel, the anchor-loop merge with the
  // token append) release their dependents only when they complete.
  pdl_launch_dependents();
  if (tid < D) q_s[tid] = __bfloat162float(a.q[(size_t)bh * D + tid]) * a.qscale;
  if (tid < kPackHeader) pack_s[tid] = 0u;
  __syncthreads();
  if (NRES > 0 && hadamard) {   // R q = H q / sqrt(128); qr_s serves as the butterflies' scratch
    float v[1] = {tid < D ? q_s[tid] : 0.f};
    hadamard128<1>(v, tid, qr_s);
    if (tid < D) qr_s[tid] = v[0];
    __syncthreads();
  } else if (NRES > 0) {   // (R q)[row] for the warp's rows: lane partials, then a reduce-scatter
    const float4 x = lane < D / 4 ? reinterpret_cast<const float4*>(q_s)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    float pv[RPW];
#pragma unroll
    for (int v = 0; v < RPW; ++v) pv[v] = fmaf(rv[v].x, x.x, fmaf(rv[v].y, x.y, fmaf(rv[v].z, x.z, rv[v].w * x.w)));
    // after the step with offset o, each lane keeps the half of its values whose
    // index bit matches its lane bit, summed with the partner's: 16 -> 8 -> 4 -> 2 -> 1
#pragma unroll
    for (int o = 16, n = RPW / 2; n >= 1; o >>= 1, n >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < n; ++i) {
        const float send = up ? pv[i] : pv[i + n];
        const float keep = up ? pv[i + n] : pv[i];
        pv[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    pv[0] += __shfl_xor_sync(0xffffffffu, pv[0], 1);
    // lanes 2v and 2v+1 now hold the sum for the warp's row index v
    const int row = warp + 8 * (lane >> 1);
    if ((lane & 1) == 0 && row < D) qr_s[row] = pv[0];
    __syncthreads();
  }
  // max |x| of each plane, and the per-group sums of x (header)
  {
    const float x0 = tid < D ? q_s[tid] : 0.f;
    const float x1 = (NRES > 0 && tid < D) ? qr_s[tid] : 0.f;
    float m0 = fabsf(x0), m1 = fabsf(x1), s0 = x0, s1 = x1;
#pragma unroll
    for (int off = GS / 2; off > 0; off >>= 1) {   // group sums: GS consecutive lanes
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    if (tid < D && tid % GS == 0) {
      pack_s[4 + tid / GS] = __float_as_uint(s0);
      pack_s[4 + NG + tid / GS] = __float_as_uint(s1);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
    }
    if (lane == 0) { red_s[0][warp] = m0; red_s[1][warp] = m1; }
  }
  __syncthreads();
  float scl[2];   // 2^k per plane
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    float mx = 0.f;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) mx = fmaxf(mx, red_s[p][w]);
    int e = 0;
    (void)frexpf(mx, &e);                  // mx = f 2^e, f in [0.5, 1)
    const int k = mx > 0.f ? 15 - e : 0;
    scl[p] = ldexpf(1.f, k);
    if (tid == 0) pack_s[p] = __float_as_uint(ldexpf(1.f, 24 - k));   // sum(code x) = D 2^(24 - k)
  }
  // the images: one thread per (piece, lane, register)
  for (int i = tid; i < 8 * NIMG; i += kPrepThreads) {
    const int piece = i / (4 * NIMG), t = (i / NIMG) % 4, rho = i % NIMG;
    uint32_t v = 0u;
    int ch[2] = {-1, -1};
    float sc = 1.f;
    bool res = false;
    if (rho < 2 * NMA) {             // anchor: word rho / 4 of the lane, register k
      const int k = rho & 3, wd = t * C::WA + (rho >> 2);
      ch[0] = 8 * wd + k;
      ch[1] = 8 * wd + k + 4;
      sc = (k & 1) ? 0.0625f : 1.f;
    } else if (t < C::TR) {          // residual: word (rho - 2 NMA) / 8 of the lane, register 2m + hb
      const int r = rho - 2 * NMA, wd = 2 * t + (r >> 3), m = (r & 7) >> 1, hb = r & 1;
      ch[0] = 16 * wd + 4 * hb + m;
      ch[1] = 16 * wd + 4 * hb + m + 8;
      sc = m == 0 ? 1.f : (m == 1 ? 0.25f : (m == 2 ? 0.0625f : 0.015625f));
      res = true;
    }
    if (ch[0] >= 0) {
      const float* xs = res ? qr_s : q_s;
      const float s = scl[res ? 1 : 0] * sc;
      __half h0, l0, h1, l1;
      f16_pieces(xs[ch[0]] * s, h0, l0);
      f16_pieces(xs[ch[1]] * s, h1, l1);
      v = piece == 0 ? pack_f16x2(h0, h1) : pack_f16x2(l0, l1);
    }
    pack_s[kPackHeader + i] = v;
  }
  __syncthreads();
  pdl_wait();   // the workspace's packs are free once the kernel ahead has finished
  uint4* dst = reinterpret_cast<uint4*>(a.packs + (size_t)bh * kPackWords);
  const uint4* src = reinterpret_cast<const uint4*>(pack_s);
  for (int i = tid; i < (kPackHeader + 8 * NIMG) / 4; i += kPrepThreads) dst[i] = src[i];
}

// PAGED: the cache uses the block-table layout (tile addresses through the table).
// Anchor-only calls: at most 72 registers, so that an append CTA of the merge
// kernel (64 registers) fits beside three decode CTAs on an SM; LEAN (64
// registers) leaves room for two, for anchor-loop calls with more append CTAs
// than SMs (their second wave would otherwise wait for the decode kernel).
template <int D, int GS, int NRES, bool PAGED, bool LEAN = false>
__global__ void __launch_bounds__(kThreads, (Cfg<D, GS, NRES>::FIT))
    __maxnreg__((LEAN ? 64 : Cfg<D, GS, NRES>::MAXREG)) decode_kernel(DecodeArgs a) {
  using C = Cfg<D, GS, NRES>;
  using LY = typename C::template Lay<PAGED>;
  constexpr int NG = C::NG, STAGES = C::STAGES, NITEM = C::NITEM, UTOK = C::UTOK;
  constexpr int NMA = C::NMA, NMR = C::NMR, NACA = C::NACA, NACR = C::NACR, NIMG = C::NIMG, NGW = C::NGW;
  constexpr typename C::AccMap MA = C::make_map(false), MR = C::make_map(true);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[STAGES];
  __shared__ int pre_s[kMaxRows + 1];
  __shared__ int nt_s[kMaxRows + 1];        // work units (128-token) per row; then a sentinel
  __shared__ int sl_s[kMaxRows];
  __shared__ __align__(16) float red_s[2][kThreads / 32];   // per-warp score maxima, by unit parity
  __shared__ float wsum_s[kThreads / 32][NITEM + 1];   // per-warp partials of off_s
  __shared__ float off_s[NITEM + 1];               // per-segment offset sums; [NITEM] = softmax sum
  uint8_t* wimg = smem + STAGES * C::STAGE;        // value-weight images, then a zero block

  pdl_launch_dependents();   // the merge kernel may start staging R
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int H = a.g.Hq, B = a.batch;   // units run over (row, query head); query head h reads KV head h / qpk
  const int Cn = gridDim.x, cta = blockIdx.x;

  // ---- per-row unit counts and prefix over (row, head) ----
  for (int b = tid; b < B; b += kThreads) {
    const int n = clamp_len(a.seq_lens[b], a.g.Nmax);
    sl_s[b] = n;
    nt_s[b] = (n + UTOK - 1) / UTOK;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      pre_s[b] = acc;
      acc += H * nt_s[b];
    }
    pre_s[B] = acc;
    nt_s[B] = 1;   // sentinel for the row walk below
  }
  __syncthreads();
  const int U = pre_s[B];

  // Every CTA waits for the kernel ahead of it before exiting, early exits
  // included, so that this kernel's completion implies the prep kernel's.
  if (U == 0) { pdl_wait(); return; }   // every row empty: the merge kernel writes the current V
  const Split split{U / Cn, U % Cn};
  const int u0 = split.start(cta), u1 = split.start(cta + 1);
  if (u0 >= u1) { pdl_wait(); return; }

  // unit cursor (row, head, unit), advanced without divisions
  struct Cursor { int b, h, t; };
  auto locate = [&](int u) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {   // last row b with pre_s[b] <= u (rows with no units are skipped)
      int mid = (lo + hi + 1) >> 1;
      if (pre_s[mid] <= u) lo = mid; else hi = mid - 1;
    }
    int rem = (int)(u - pre_s[lo]);
    return Cursor{lo, rem / nt_s[lo], rem % nt_s[lo]};
  };
  auto advance = [&](Cursor& c) {
    if (++c.t == nt_s[c.b]) {
      c.t = 0;
      if (++c.h == H) {
        c.h = 0;
        do { ++c.b; } while (nt_s[c.b] == 0);   // nt_s[B] = 1 stops the walk
      }
    }
  };
  // producer cursor (thread 0 only), in shared memory: it costs the other threads no registers
  __shared__ Cursor pc;
  if (tid == 0) pc = locate(u0);
  const uint64_t pol = l2_evict_first_policy();   // the cache is read once per call
  // layout tiles of the producer's unit that hold tokens (the last unit of a row may have one)
  auto unit_tiles = [&]() { return min(C::UT, (sl_s[pc.b] - pc.t * C::UT * kTile + kTile - 1) / kTile); };
  // paged layout: block-table entries of the next unit's tiles, fetched one unit
  // ahead by the producer thread with asynchronous copies, so that neither the
  // copies nor the producer's own unit wait on them (kept in shared memory: the
  // producer's state costs the other threads no registers)
  __shared__ int next_raw_s[C::UT];
  __shared__ int pu_s;   // unit the producer issues next
  auto fetch_pages = [&]() {
    const int nt = unit_tiles();
#pragma unroll
    for (int k = 0; k < C::UT; ++k) {
      if (k < nt)
        cp_async4(&next_raw_s[k], a.g.table + (size_t)pc.b * a.g.max_tiles + pc.t * C::UT + k);
      else
        next_raw_s[k] = 0;
    }
    cp_async_commit();
  };
  auto issue = [&](int stage) {
    if constexpr (PAGED) cp_async_wait_all();   // this unit's entries (fetched an issue ago)
    const int t0 = pc.t * C::UT;
    const int ntile = unit_tiles();
    const int kvh = pc.h / a.g.qpk;
    const uint8_t* region = PAGED ? a.base : a.base + a.g.region_offset(a.layer, a.group, pc.b, kvh);
    uint8_t* dst = smem + stage * C::STAGE;
    mbar_arrive_expect_tx(&full_bar[stage], (uint32_t)(ntile * C::SUB));
    // plane slots of the stage: K anchor, V anchor, then K and V of each residual plane
    auto slot = [&](bool anchor, int r, int kv) {
      return dst + (anchor ? kv * C::PA : 2 * C::PA + (2 * r + kv) * C::PR);
    };
    if constexpr (PAGED) {
      for (int k = 0; k < ntile; ++k) {   // a tile per page: anchor pair, then the residual planes read
        const int page = max(checked_page(a.g, next_raw_s[k], a.status), 0);   // a bad entry reads page 0
        // this head's block of the tile's page (same offsets as Geom::tile_offset, sizes as constants)
        const uint8_t* blk = a.base + (((int64_t)a.layer * a.g.G + a.group) * a.g.num_pages + page) * a.g.page_bytes +
                             (int64_t)kvh * a.g.head_block;
        uint8_t* d = dst + k * C::SUB;
        bulk_g2s_hint(d, blk, 2 * C::A_TILE, &full_bar[stage], pol);
        if constexpr (NRES > 0)
          bulk_g2s_hint(d + 2 * C::A_TILE, blk + 2 * C::A_TILE + 2 * a.res0 * C::R_TILE, 2 * NRES * C::R_TILE,
                        &full_bar[stage], pol);
      }
    } else {   // the unit's tiles of a plane are contiguous: one copy per plane
      const uint32_t na = (uint32_t)(ntile * C::A_TILE), nr = (uint32_t)(ntile * C::R_TILE);
      bulk_g2s_hint(slot(true, 0, 0), region + a.g.anchor_plane(0) + (int64_t)t0 * C::A_TILE, na, &full_bar[stage], pol);
      bulk_g2s_hint(slot(true, 0, 1), region + a.g.anchor_plane(1) + (int64_t)t0 * C::A_TILE, na, &full_bar[stage], pol);
#pragma unroll
      for (int r = 0; r < NRES; ++r) {
        bulk_g2s_hint(slot(false, r, 0), region + a.g.res_plane(a.res0 + r, 0) + (int64_t)t0 * C::R_TILE, nr,
                      &full_bar[stage], pol);
        bulk_g2s_hint(slot(false, r, 1), region + a.g.res_plane(a.res0 + r, 1) + (int64_t)t0 * C::R_TILE, nr,
                      &full_bar[stage], pol);
      }
    }
    advance(pc);
    if constexpr (PAGED)
      if (++pu_s < u1) fetch_pages();
  };

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&full_bar[s], 1);
    fence_mbar_init();
  }
  // the zero block that idle lanes read their value B operands from
  for (int i = tid; i < 64; i += kThreads) reinterpret_cast<uint32_t*>(wimg + NITEM * kWItem)[i] = 0u;
  __syncthreads();
  if (tid == 0) {
    if constexpr (PAGED) {
      pu_s = u0;
      fetch_pages();
    }
    for (int s = 0; s < STAGES && u0 + s < u1; ++s) issue(s);
  }
  Cursor cc = locate(u0);   // consumer cursor
  pdl_wait();               // the query packs of qprep_kernel are complete

  // ---- per-thread constants ----
  // scoring: rows gid and gid + 8 of the warp's products are tokens tk0 and tk0 + 2
  // (tk0 = 16 warp + 4 (gid / 2) + gid % 2; rows r0, r0 + 2 of tile tau), the pair
  // that one f16x2 operand of the value products holds
  const int tk0 = 16 * warp + 4 * (gid >> 1) + (gid & 1), tau = warp >> 2, r0 = tk0 & (kTile - 1);
  // value-weight slot of the pair in the INT4 (anchor) and INT2 (residual) images
  int so4, so2;
  float sc4, sc2;
  int4_slot(tk0, so4, sc4);
  int2_slot(tk0, so2, sc2);
  const bool bq_lane = (gid >> 1) == tig;   // lanes whose scoring B operands are not zero
  // value products: channels vc0 = 16 warp + gid, vc1 = vc0 + 8 of group vg
  const bool v_act = warp < C::VW;
  const int vc0 = 16 * warp + gid, vg = (16 * warp) / GS;
  const uint8_t* vzero = wimg + NITEM * kWItem;

  // ---- per-segment state ----
  uint32_t bq[NIMG];                 // B operands of the scoring products (query, rotated query)
  float sig_a = 0.f, sig_r = 0.f;
  float qa_own[NACA], qr_own[NACR];  // the offset sums of the groups this lane adds
  float acc_a[4] = {0.f, 0.f, 0.f, 0.f}, acc_r[4] = {0.f, 0.f, 0.f, 0.f};   // value accumulators (d0..d3 of the value products)
  float m_run = -INFINITY;
  float off_part[1 + NRES][NGW];     // partial offset sums of this lane's weight groups
  float l_part = 0.f;                // partial softmax denominator (lanes tig == 0)
  int cur_bh = -1;
  bool aborted = false;
  int fail_u = 0;

  auto flush = [&](int bh) {
    // finish the segment's partials: offset sums per item and the softmax
    // denominator, per warp, then over the warps in a fixed order (repeated calls
    // give equal bits)
#pragma unroll
    for (int j = 0; j <= NRES; ++j)
#pragma unroll
      for (int s = 0; s < NGW; ++s) {
        float x = off_part[j][s];
        for (int off = 4; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        const int g = tig + 4 * s;
        if (gid == 0 && g < NG) wsum_s[warp][j * NG + g] = x;
      }
    {
      float x = l_part;
      for (int off = 4; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      if (lane == 0) wsum_s[warp][NITEM] = x;
    }
    __syncthreads();
    for (int i = tid; i <= NITEM; i += kThreads) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) x += wsum_s[w][i];
      off_s[i] = x;
    }
    __syncthreads();
    // this CTA's partial for bh; merge_kernel combines the partials
    float* part = a.partials + (size_t)(cta + bh) * a.pstride;
    if (tid == 0) {
      part[0] = m_run;
      part[1] = off_s[NITEM];
    }
    if (v_act && tig == 0) {
      float oa = off_s[vg], orr = 0.f;
#pragma unroll
      for (int r = 0; r < NRES; ++r) orr += off_s[(1 + r) * NG + vg];
      part[2 + vc0] = fmaf(acc_a[0] + acc_a[1], 16777216.f, oa);
      part[2 + vc0 + 8] = fmaf(acc_a[2] + acc_a[3], 16777216.f, oa);
      if (NRES > 0) {
        part[2 + D + vc0] = fmaf(acc_r[0] + acc_r[1], 16777216.f, orr);
        part[2 + D + vc0 + 8] = fmaf(acc_r[2] + acc_r[3], 16777216.f, orr);
      }
    }
  };

  auto begin_segment = [&](int bh) {
    const uint32_t* pk = a.packs + (size_t)bh * kPackWords;
    sig_a = __uint_as_float(__ldcg(pk + 0));
    sig_r = __uint_as_float(__ldcg(pk + 1));
#pragma unroll
    for (int ac = 0; ac < NACA; ++ac) qa_own[ac] = __uint_as_float(__ldcg(pk + 4 + C::ga(tig, MA.rep[ac])));
#pragma unroll
    for (int ac = 0; ac < NACR; ++ac)
      qr_own[ac] = tig < C::TR ? __uint_as_float(__ldcg(pk + 4 + NG + C::gr(tig, MR.rep[ac]))) : 0.f;
    // the image of this lane (piece gid & 1, lane tig), when it is one of the eight non-zero ones
    const uint4* img = reinterpret_cast<const uint4*>(pk + kPackHeader + ((gid & 1) * 4 + tig) * NIMG);
#pragma unroll
    for (int i = 0; i < NIMG / 4; ++i) {
      const uint4 v = bq_lane ? __ldcg(img + i) : make_uint4(0u, 0u, 0u, 0u);
      bq[4 * i] = v.x; bq[4 * i + 1] = v.y; bq[4 * i + 2] = v.z; bq[4 * i + 3] = v.w;
    }
    m_run = -INFINITY;
    l_part = 0.f;
#pragma unroll
    for (int j = 0; j <= NRES; ++j)
#pragma unroll
      for (int s = 0; s < NGW; ++s) off_part[j][s] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) { acc_a[i] = 0.f; acc_r[i] = 0.f; }
    cur_bh = bh;
  };

  for (int u = u0; u < u1; ++u, advance(cc)) {
    const int it = (int)(u - u0), stage = it % STAGES, buf = it & 1;
    const int bh = cc.b * H + cc.h;
    if (bh != cur_bh) {
      if (cur_bh >= 0) flush(cur_bh);
      begin_segment(bh);
    }
    const int n_valid = min(UTOK, sl_s[cc.b] - cc.t * UTOK);

    if (!mbar_wait_bounded(&full_bar[stage], (uint32_t)((it / STAGES) & 1))) aborted = true;

    const uint8_t* st = smem + stage * C::STAGE;
    // this lane's tokens: tile tau of each plane
    const uint8_t* sak = st + tau * LY::TA;                 // K anchor
    const uint8_t* sav = st + LY::AV + tau * LY::TA;        // V anchor
    const uint8_t* sres = st + LY::RB + tau * LY::TR;       // + (2 r + kv) PL: residual plane r

    // ---- scores of tokens tk0, tk1: tensor-core products over the K planes ----
    float sc0, sc1;
    {
      // anchor: this lane's words of the two token rows
      uint32_t wa0[C::WA], wa1[C::WA];
      const uint8_t* ak = sak + r0 * (D / 2) + tig * (D / 8);
      if constexpr (C::WA == 4) {
        const uint4 x0 = *reinterpret_cast<const uint4*>(ak);
        const uint4 x1 = *reinterpret_cast<const uint4*>(ak + 2 * (D / 2));
        wa0[0] = x0.x; wa0[1] = x0.y; wa0[2] = x0.z; wa0[3] = x0.w;
        wa1[0] = x1.x; wa1[1] = x1.y; wa1[2] = x1.z; wa1[3] = x1.w;
      } else {
#pragma unroll
        for (int k = 0; k < C::WA; ++k) {
          wa0[k] = *reinterpret_cast<const uint32_t*>(ak + 4 * k);
          wa1[k] = *reinterpret_cast<const uint32_t*>(ak + 2 * (D / 2) + 4 * k);
        }
      }
      float da[NACA][4];
#pragma unroll
      for (int ac = 0; ac < NACA; ++ac) da[ac][0] = da[ac][1] = da[ac][2] = da[ac][3] = 0.f;
#pragma unroll
      for (int k = 0; k < C::WA; ++k) {
        uint32_t x0[4], x1[4];
        int4_f16(wa0[k], x0);
        int4_f16(wa1[k], x1);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * k + jj;
          mma16816(da[MA.acc[j]], x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1], bq[2 * j], bq[2 * j + 1]);
        }
      }
      // anchor score per token: sum over this lane's accumulators of s * (dot product) + o * sum(q)
      float sa0 = 0.f, sa1 = 0.f;
      const uint8_t* am = sak + C::A_CODES + r0 * NG * 2;
#pragma unroll
      for (int ac = 0; ac < NACA; ++ac) {
        const int g = C::ga(tig, MA.rep[ac]);
        const float2 m0 = meta2(am + g * 2), m1 = meta2(am + 2 * NG * 2 + g * 2);
        const bool own = (MA.own >> (4 * ac + tig)) & 1u;
        sa0 = fmaf(m0.x, (da[ac][0] + da[ac][1]) * sig_a, own ? fmaf(m0.y, qa_own[ac], sa0) : sa0);
        sa1 = fmaf(m1.x, (da[ac][2] + da[ac][3]) * sig_a, own ? fmaf(m1.y, qa_own[ac], sa1) : sa1);
      }
      sc0 = sa0;
      sc1 = sa1;
      if constexpr (NRES > 0) {
        float cp0 = 1.f, cp1 = 1.f, sr0 = 0.f, sr1 = 0.f;
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const uint8_t* rk = sres + 2 * r * LY::PL;
          float dr[NACR][4];
#pragma unroll
          for (int ac = 0; ac < NACR; ++ac) dr[ac][0] = dr[ac][1] = dr[ac][2] = dr[ac][3] = 0.f;
          // lanes without residual words (d = 96: lane 3) take part with zero operands:
          // the products are warp-wide
          uint32_t w0[2] = {0u, 0u}, w1[2] = {0u, 0u};
          if (tig < C::TR) {
            const uint8_t* rr = rk + r0 * (D / 4) + tig * 8;
            const uint2 y0 = *reinterpret_cast<const uint2*>(rr);
            const uint2 y1 = *reinterpret_cast<const uint2*>(rr + 2 * (D / 4));
            w0[0] = y0.x; w0[1] = y0.y; w1[0] = y1.x; w1[1] = y1.y;
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t x0[8], x1[8];
            int2_f16(w0[k], x0);
            int2_f16(w1[k], x1);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int j = 4 * k + jj;
              mma16816(dr[MR.acc[j]], x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1],
                       bq[2 * NMA + 2 * j], bq[2 * NMA + 2 * j + 1]);
            }
          }
          float s0 = 0.f, s1 = 0.f;
          if (tig < C::TR) {
            const uint8_t* rm = rk + C::R_CODES + r0 * NG * 2;
#pragma unroll
            for (int ac = 0; ac < NACR; ++ac) {
              const int g = C::gr(tig, MR.rep[ac]);
              const float2 m0 = meta2(rm + g * 2), m1 = meta2(rm + 2 * NG * 2 + g * 2);
              const bool own = (MR.own >> (4 * ac + tig)) & 1u;
              s0 = fmaf(m0.x, (dr[ac][0] + dr[ac][1]) * sig_r, own ? fmaf(m0.y, qr_own[ac], s0) : s0);
              s1 = fmaf(m1.x, (dr[ac][2] + dr[ac][3]) * sig_r, own ? fmaf(m1.y, qr_own[ac], s1) : s1);
            }
          }
          const uint8_t* rc = rk + C::R_CODES + C::META + r0 * 2;
          const float c0 = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc));
          const float c1 = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc + 4));
          // chained: plane r weighs the product of the coefficients before it
          sr0 = fmaf(cp0, s0, sr0);
          sr1 = fmaf(cp1, s1, sr1);
          cp0 *= c0;
          cp1 *= c1;
        }
        sc0 = fmaf(cp0, sa0, sr0);
        sc1 = fmaf(cp1, sa1, sr1);
      }
      // the token's score: the sum over the four lanes of its row
      sc0 += __shfl_xor_sync(0xffffffffu, sc0, 1);
      sc1 += __shfl_xor_sync(0xffffffffu, sc1, 1);
      sc0 += __shfl_xor_sync(0xffffffffu, sc0, 2);
      sc1 += __shfl_xor_sync(0xffffffffu, sc1, 2);
    }
    const bool ok0 = !aborted && tk0 < n_valid, ok1 = !aborted && tk0 + 2 < n_valid;
    if (!ok0) sc0 = -INFINITY;
    if (!ok1) sc1 = -INFINITY;
    float wmax = fmaxf(sc0, sc1);
    for (int off = 4; off < 32; off <<= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
    if (lane == 0) red_s[buf][warp] = wmax;
    if (__syncthreads_or(aborted)) {                   // B1: per-warp score maxima are in red_s
      fail_u = u;
      aborted = true;
      if (tid == 0) atomicExch(&a.status[0], 1);
      break;
    }
    // every warp has finished the previous unit: its stage can be refilled
    if (tid == 0 && it >= 1 && u - 1 + STAGES < u1) issue((it - 1) % STAGES);

    const float4 ma4 = reinterpret_cast<const float4*>(red_s[buf])[0], mb4 = reinterpret_cast<const float4*>(red_s[buf])[1];
    const float m_tile = fmaxf(fmaxf(fmaxf(ma4.x, ma4.y), fmaxf(ma4.z, ma4.w)), fmaxf(fmaxf(mb4.x, mb4.y), fmaxf(mb4.z, mb4.w)));
    const float m_new = fmaxf(m_run, m_tile);
    const float alpha = ex2_fast(m_run - m_new);   // 0 on the first unit (m_run = -inf)
    m_run = m_new;

    // ---- value weights p * coefficients * scale of this lane's (token, group)
    //      pairs as f16 pieces into the images; offsets p * coefficients * offset ----
    const float p0 = ex2_fast(sc0 - m_new), p1 = ex2_fast(sc1 - m_new);   // 0 for masked tokens
    if (tig == 0) l_part = fmaf(l_part, alpha, p0 + p1);
#pragma unroll
    for (int j = 0; j <= NRES; ++j)
#pragma unroll
      for (int s = 0; s < NGW; ++s) off_part[j][s] *= alpha;
#pragma unroll
    for (int s = 0; s < NGW; ++s) {
      const int g = tig + 4 * s;
      if (g < NG) {
        float cp0 = p0, cp1 = p1;   // p times the coefficients of the planes before the current one
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const uint8_t* rv = sres + (2 * r + 1) * LY::PL + C::R_CODES;
          const float2 v0 = meta2(rv + r0 * NG * 2 + g * 2), v1 = meta2(rv + (r0 + 2) * NG * 2 + g * 2);
          if (ok0) off_part[1 + r][s] = fmaf(cp0, v0.y, off_part[1 + r][s]);
          if (ok1) off_part[1 + r][s] = fmaf(cp1, v1.y, off_part[1 + r][s]);
          uint32_t hi, lo;
          f16x2_pieces(ok0 ? cp0 * v0.x * sc2 : 0.f, ok1 ? cp1 * v1.x * sc2 : 0.f, hi, lo);
          uint8_t* im = wimg + ((1 + r) * NG + g) * kWItem + so2;
          *reinterpret_cast<uint32_t*>(im) = hi;
          *reinterpret_cast<uint32_t*>(im + kWPiece) = lo;
          const uint8_t* rc = rv + C::META + r0 * 2;
          if (ok0) cp0 *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc));
          if (ok1) cp1 *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc + 4));
        }
        const uint8_t* am = sav + C::A_CODES;
        const float2 a0 = meta2(am + r0 * NG * 2 + g * 2), a1 = meta2(am + (r0 + 2) * NG * 2 + g * 2);
        if (ok0) off_part[0][s] = fmaf(cp0, a0.y, off_part[0][s]);
        if (ok1) off_part[0][s] = fmaf(cp1, a1.y, off_part[0][s]);
        uint32_t hi, lo;
        f16x2_pieces(ok0 ? cp0 * a0.x * sc4 : 0.f, ok1 ? cp1 * a1.x * sc4 : 0.f, hi, lo);
        uint8_t* im = wimg + g * kWItem + so4;
        *reinterpret_cast<uint32_t*>(im) = hi;
        *reinterpret_cast<uint32_t*>(im + kWPiece) = lo;
      }
    }
    __syncthreads();                                   // B2: the weight images are complete

    // ---- value products: channels vc0, vc0 + 8 against the weights of the 128 tokens ----
    if (v_act) {
      const uint8_t* vb = gid < 2 ? wimg + vg * kWItem + gid * kWPiece + tig * 8 : vzero + tig * 8;
      float dv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int t2 = 0; t2 < C::UT; ++t2) {
        const uint8_t* av = st + LY::AV + t2 * LY::TA + vc0 * (kTile / 2) + tig * 8;
        const uint2 y0 = *reinterpret_cast<const uint2*>(av);
        const uint2 y1 = *reinterpret_cast<const uint2*>(av + 8 * (kTile / 2));
        const uint32_t w0[2] = {y0.x, y0.y}, w1[2] = {y1.x, y1.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t x0[4], x1[4];
          int4_f16(w0[e], x0);
          int4_f16(w1[e], x1);
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int m = 2 * (2 * t2 + e) + jj;
            const uint2 bb = *reinterpret_cast<const uint2*>(vb + m * 32);
            mma16816(dv, x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1], bb.x, bb.y);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) acc_a[i] = fmaf(acc_a[i], alpha, dv[i]);
      if constexpr (NRES > 0) {
        float dr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const uint8_t* vbr = gid < 2 ? wimg + ((1 + r) * NG + vg) * kWItem + gid * kWPiece + tig * 8 : vzero + tig * 8;
#pragma unroll
          for (int t2 = 0; t2 < C::UT; ++t2) {
            const uint8_t* rvp = st + LY::RB + (2 * r + 1) * LY::PL + t2 * LY::TR + vc0 * (kTile / 4) + tig * 4;
            const uint32_t y0 = *reinterpret_cast<const uint32_t*>(rvp);
            const uint32_t y1 = *reinterpret_cast<const uint32_t*>(rvp + 8 * (kTile / 4));
            uint32_t x0[8], x1[8];
            int2_f16(y0, x0);
            int2_f16(y1, x1);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int m = 4 * t2 + jj;
              const uint2 bb = *reinterpret_cast<const uint2*>(vbr + m * 32);
              mma16816(dr, x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1], bb.x, bb.y);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc_r[i] = fmaf(acc_r[i], alpha, dr[i]);
      }
    }
    // no barrier here: the next unit writes the images only after its B1, and its
    // stage is refilled after the next B1
  }

  if (aborted) {
    // let the copies still in flight land before the CTA exits (each wait bounded)
    if (tid == 0) {
      for (int v = fail_u; v < u1 && v < fail_u + STAGES; ++v)
        (void)mbar_wait_bounded(&full_bar[(v - u0) % STAGES], (uint32_t)(((v - u0) / STAGES) & 1));
      if constexpr (PAGED) cp_async_wait_all();   // block-table entries fetched ahead
    }
    __syncthreads();
    return;
  }
  __syncthreads();
  if (cur_bh >= 0) flush(cur_bh);
  (void)NMR;
}

// Combines the partial softmax states of (row, head) blockIdx.x: the CTAs that
// held its units are recomputed from seq_lens with the decode kernel's split.
// APPEND (anchor-loop call only): the grid has two CTAs per (row, head); they
// also compress the current token's K (first CTA, which also merges) and V
// (second CTA) into the cache at position seq_lens[row] (rq_token_append.cuh).
// They run 128 threads of at most 64 registers: one such CTA fits beside three
// anchor-call decode CTAs (72 registers each) and does that work while they stream.
template <int D, int NRES, bool APPEND>
__global__ void __launch_bounds__(APPEND ? kAppendThreads : kMergeThreads, APPEND ? 8 : 0)
    merge_kernel(DecodeArgs a, int Cn) {
  static_assert(!APPEND || NRES == 0, "append runs in the anchor-loop merge");
  constexpr int NT = APPEND ? kAppendThreads : kMergeThreads;
  static_assert(NRES == 0 ? NT >= D : NT >= 2 * D, "a thread per accumulator element");
  extern __shared__ __align__(16) float R_s[];   // [D][D] when NRES > 0; the append's scratch with APPEND
  __shared__ float w_s[NRES == 0 ? 1 : kMaxContrib];   // contributor weights (residual-loop merges)
  __shared__ float l_s[NRES == 0 ? 1 : kMaxContrib];
  __shared__ float ml_s[2];
  __shared__ float va_s[D];
  __shared__ __align__(16) float vr_s[D];
  __shared__ float rt_s[D];
  __shared__ float redf_s[NT / 32];
  __shared__ int redi_s[2][NT / 32];
  __shared__ uint64_t r_bar;
  constexpr int UTOK = 2 * kTile;
  // the next call's prep may start loading R (it waits for this kernel); the
  // appending variant writes the cache, so its dependents wait for it to finish
  if constexpr (!APPEND) pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.g.Hq, B = a.batch, Hkv = a.g.H;   // merge CTAs: one per (row, query head)
  // APPEND: CTAs [0, B*Hq) merge, the first query head of each KV head also coding
  // the token's K; CTAs [B*Hq, B*Hq + B*Hkv) code the V of one (row, KV head).
  // With several query heads per KV head the coding CTAs come first instead, so
  // that they take the SM room beside the decode kernel before the merge-only
  // ones: [0, B*Hkv) code V, [B*Hkv, 2 B*Hkv) merge the first query head of each
  // KV head and code its K, the rest merge the other query heads (ouro8k batch 4
  // with 64 query heads: anchor-loop call 48.3 -> 42.2 us).
  const int qpk = a.g.qpk;
  const bool coders_first = APPEND && qpk > 1;
  const bool v_cta = APPEND && (coders_first ? (int)blockIdx.x < B * Hkv : (int)blockIdx.x >= B * H);
  int bh, b, h, kvh;
  if (!coders_first) {
    if (v_cta) {
      const int r = blockIdx.x - B * H;
      b = r / Hkv;
      kvh = r - b * Hkv;
      h = kvh * qpk;
      bh = b * H + h;
    } else {
      bh = blockIdx.x;
      b = bh / H;
      h = bh - b * H;
      kvh = h / qpk;
    }
  } else {
    int r = blockIdx.x;
    if (r < 2 * B * Hkv) {   // V coder, or first query head of its KV head (K coder)
      r = r < B * Hkv ? r : r - B * Hkv;
      b = r / Hkv;
      kvh = r - b * Hkv;
      h = kvh * qpk;
    } else {                 // query heads 1 .. qpk-1 of each KV head
      r -= 2 * B * Hkv;
      const int per_row = Hkv * (qpk - 1);
      b = r / per_row;
      const int rem = r - b * per_row;
      kvh = rem / (qpk - 1);
      h = kvh * qpk + 1 + (rem - kvh * (qpk - 1));
    }
    bh = b * H + h;
  }
  const int kvbh = b * Hkv + kvh;   // the current token's K/V are per KV head

  // ---- before the wait: inputs the decode kernel does not write ----
  const bool hadamard = (a.g.mode & RQ_MODE_HADAMARD) != 0;   // R^T as the fast transform (d = 128)
  bool app_ok = false;
  int app_pos = 0, app_page = 0;
  uint8_t* app_smem = reinterpret_cast<uint8_t*>(R_s);
  if constexpr (APPEND) {
    if (v_cta || h % a.g.qpk == 0) {   // the same for every thread of the CTA
      app_pos = a.seq_lens[b];
      app_ok = token_append_compute<D>(a.g, const_cast<uint8_t*>(a.base), a.R, a.kv_all, B, a.layer, a.group, b,
                                       kvh, v_cta ? 1 : 0, app_pos, a.status, app_smem, &app_page);
    }
    if (v_cta) {   // store after the wait; the merge CTAs merge
      pdl_wait();
      if (app_ok)
        token_append_store<D>(a.g, const_cast<uint8_t*>(a.base), a.layer, a.group, b, kvh, 1, app_pos, app_page,
                              app_smem);
      return;
    }
  }
  if (NRES > 0 && !hadamard && tid == 0) {   // R -> shared memory, one bulk copy (R is 16-byte aligned)
    mbar_init(&r_bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&r_bar, (uint32_t)(D * D * sizeof(float)));
    bulk_g2s(R_s, a.R, (uint32_t)(D * D * sizeof(float)), &r_bar);
  }
  // the current token's value element of this thread (an input: read before the wait)
  const float vcur = tid < D ? __bfloat162float(a.v_cur[(size_t)kvbh * D + tid]) : 0.f;
  // current token's score (base 2)
  float sc = 0.f;
  for (int k = tid; k < D; k += NT)
    sc += __bfloat162float(a.q[(size_t)bh * D + k]) * a.qscale *
          __bfloat162float(a.k_cur[(size_t)kvbh * D + k]);
  // units before this row and in total (same clamping and unit size as the decode kernel)
  int before = 0, total = 0;
  for (int r = tid; r < B; r += NT) {
    const int nt = (clamp_len(a.seq_lens[r], a.g.Nmax) + UTOK - 1) / UTOK;
    total += (H / a.qh) * nt;
    if (r < b) before += (H / a.qh) * nt;
  }
  for (int off = 16; off > 0; off >>= 1) {
    sc += __shfl_xor_sync(0xffffffffu, sc, off);
    before += __shfl_xor_sync(0xffffffffu, before, off);
    total += __shfl_xor_sync(0xffffffffu, total, off);
  }
  if (lane == 0) { redf_s[warp] = sc; redi_s[0][warp] = before; redi_s[1][warp] = total; }
  __syncthreads();
  float s_cur = 0.f;
  int pre = 0, U = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) { s_cur += redf_s[w]; pre += redi_s[0][w]; U += redi_s[1][w]; }
  const int ntb = (clamp_len(a.seq_lens[b], a.g.Nmax) + UTOK - 1) / UTOK;
  if (ntb == 0) {   // empty cache: attention over the current token alone
    if (NRES > 0 && !hadamard) (void)mbar_wait_bounded(&r_bar, 0);   // the R copy lands before the CTA exits
    pdl_wait();   // completion of this kernel implies the decode kernel's
    // written after the wait: the previous call's merge may still write its output
    if (tid < D) a.out[(size_t)bh * D + tid] = vcur;
    if constexpr (APPEND)
      if (app_ok)
        token_append_store<D>(a.g, const_cast<uint8_t*>(a.base), a.layer, a.group, b, kvh, 0, app_pos, app_page,
                              app_smem);
    return;
  }
  const Split split{U / Cn, U % Cn};
  const int s0 = pre + (h / a.qh) * ntb, s1 = s0 + ntb;   // the units of h's head group
  const int c_lo = split.owner(s0), c_hi = split.owner(s1 - 1);
  const int nc = min(c_hi - c_lo + 1, kMaxContrib);

  pdl_wait();   // every partial of the decode kernel is written and visible
  if constexpr (APPEND)   // no kernel before this one is running: the new slot can be written
    if (app_ok)
      token_append_store<D>(a.g, const_cast<uint8_t*>(a.base), a.layer, a.group, b, kvh, 0, app_pos, app_page,
                            app_smem);

  // The combine, in batches of PF contributors (one L2 round trip per batch).
  // PF = 16: a (row, head) of 128 units (16k tokens) at batch 2 has about 15
  // contributors, one batch (8 in flight took two round trips there: ouro16k b2
  // step 3.25 against 3.14 ms; 32 gave 3.21 ms).
  constexpr int PF = 16;
  const bool acc_thread = tid < (NRES > 0 ? 2 * D : D);   // NT covers them (static_assert above)
  // contributor i's partial for this head: row (c_lo + i + group) * qh + (h mod qh),
  // group = the head's (row, head group) index (qh = 1: row c_lo + i + bh)
  const int hgq = b * (H / a.qh) + h / a.qh;
  const float* pbase = a.partials + ((size_t)(c_lo + hgq) * a.qh + h % a.qh) * a.pstride;
  const size_t cstride = (size_t)a.qh * a.pstride;
  const float* pc = pbase + 2 + tid;
  float L = 0.f;
  if constexpr (NRES == 0) {
    // Anchor-loop merges, with and without the append (the two must agree bit
    // for bit): every warp combines the contributors itself.  Lane k reads
    // contributor k's (m, l), the maximum and the softmax sum are taken across
    // the lanes, and each lane's weight reaches the others by shuffles.  No
    // shared memory for the weights: the appending CTA stays small enough to
    // start beside the decode CTAs.  (In the residual-loop merge, eight warps
    // redoing this cost more than the barrier it saves.)
    if (acc_thread) {   // whole warps (2D or D threads)
      float M = s_cur, v = 0.f;   // running maximum; L and v are relative to it
#pragma unroll 1
      for (int i0 = 0; i0 < nc; i0 += PF) {
        float x[PF];
#pragma unroll
        for (int k = 0; k < PF; ++k) x[k] = i0 + k < nc ? __ldcg(pc + (size_t)(i0 + k) * cstride) : 0.f;
        const float2 ml = lane < PF && i0 + lane < nc
                              ? __ldcg(reinterpret_cast<const float2*>(pbase + (size_t)(i0 + lane) * cstride))
                              : make_float2(-INFINITY, 0.f);
        float Mb = fmaxf(M, ml.x);
        for (int off = 16; off > 0; off >>= 1) Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, off));
        const float r = exp2f(M - Mb);
        M = Mb;
        const float wl = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);   // lane's contributor weight
        float lsum = wl * ml.y;
        for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        L = fmaf(L, r, lsum);
        v *= r;
#pragma unroll
        for (int k = 0; k < PF; ++k) v = fmaf(__shfl_sync(0xffffffffu, wl, k), x[k], v);   // contributor order
      }
      const float wc = exp2f(s_cur - M);   // the current token
      L += wc;
      if (tid < D) va_s[tid] = fmaf(wc, vcur, v);
      else vr_s[tid - D] = v;
    }
  } else {
    // warp 0 reads the (m, l) pairs and parks the weights in shared memory while
    // every thread loads its element of the first PF contributors' accumulators
    float xa[PF];
#pragma unroll
    for (int k = 0; k < PF; ++k) xa[k] = (acc_thread && k < nc) ? __ldcg(pc + (size_t)k * cstride) : 0.f;
    if (warp == 0) {
      // (m, l) of each contributor, read once: m parked in w_s, l in l_s
      float M = s_cur;
      for (int i = lane; i < nc; i += 32) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(pbase + (size_t)i * cstride));
        w_s[i] = ml.x;
        l_s[i] = ml.y;
        M = fmaxf(M, ml.x);
      }
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      float L = 0.f;
      for (int i = lane; i < nc; i += 32) {
        const float w = exp2f(w_s[i] - M);
        w_s[i] = w;
        L = fmaf(w, l_s[i], L);
      }
      for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
      if (lane == 0) { ml_s[0] = M; ml_s[1] = L + exp2f(s_cur - M); }
    }
    __syncthreads();
    const float M = ml_s[0];
    L = ml_s[1];
    // thread = (channel, anchor | residual accumulator)
    if (acc_thread) {
      float v = 0.f;
#pragma unroll
      for (int k = 0; k < PF; ++k)
        if (k < nc) v = fmaf(w_s[k], xa[k], v);
      // the rest in batches of PF independent loads (one L2 round trip per batch),
      // summed in contributor order as above
      for (int i0 = PF; i0 < nc; i0 += PF) {
        float x[PF];
#pragma unroll
        for (int k = 0; k < PF; ++k) x[k] = i0 + k < nc ? __ldcg(pc + (size_t)(i0 + k) * cstride) : 0.f;
#pragma unroll
        for (int k = 0; k < PF; ++k)
          if (i0 + k < nc) v = fmaf(w_s[i0 + k], x[k], v);
      }
      if (tid < D) va_s[tid] = fmaf(exp2f(s_cur - M), vcur, v);
      else vr_s[tid - D] = v;
    }
  }
  __syncthreads();
  float o = 0.f;
  if (NRES > 0 && hadamard) {
    float v[1] = {tid < D ? vr_s[tid] : 0.f};
    hadamard128<1>(v, tid, rt_s);
    o = v[0];
  } else if (NRES > 0) {
    // R in shared memory (bounded wait; a timeout sets the status word, decided for the CTA)
    const bool ok = mbar_wait_bounded(&r_bar, 0);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicExch(&a.status[0], 1);
      return;
    }
    // (R^T acc_r)[c]: thread = (column c, half of the rows), four accumulator chains
    if (tid < 2 * D) {
      const int c = tid % D, hh = tid / D;
      const float* rc = R_s + (size_t)hh * (D / 2) * D + c;
      const float* vr = vr_s + hh * (D / 2);
      float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
#pragma unroll 4
      for (int k = 0; k < D / 2; k += 4) {
        const float4 x = *reinterpret_cast<const float4*>(vr + k);
        t0 = fmaf(rc[(k + 0) * D], x.x, t0);
        t1 = fmaf(rc[(k + 1) * D], x.y, t1);
        t2 = fmaf(rc[(k + 2) * D], x.z, t2);
        t3 = fmaf(rc[(k + 3) * D], x.w, t3);
      }
      o = (t0 + t1) + (t2 + t3);
      if (hh == 1) rt_s[c] = o;
    }
    __syncthreads();
    if (tid < D) o += rt_s[tid];
  }
  if (tid < D) a.out[(size_t)bh * D + tid] = (va_s[tid] + o) / L;
}

template <int D, int GS, int NRES, bool PAGED>
cudaError_t launch_t(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  using C = Cfg<D, GS, NRES>;
  auto k = decode_kernel<D, GS, NRES, PAGED>;
  auto km = merge_kernel<D, (NRES > 0 ? 1 : 0), false>;
  const int bhs = a.batch * a.g.Hq;   // (row, query head) pairs
  size_t km_smem = NRES > 0 ? (size_t)D * D * sizeof(float) : 0;
  if (a.g.mode & RQ_MODE_HADAMARD) km_smem = 0;   // no R to stage
  int km_threads = kMergeThreads, km_extra = 0;
  if constexpr (NRES == 0)
    if (a.kv_all) {
      km = merge_kernel<D, 0, true>;
      km_smem = TokenAppendSmem::bytes(a.g.P);
      km_threads = kAppendThreads;
      km_extra = a.batch * a.g.H;   // the V-coding CTAs, one per (row, KV head)
      // more append CTAs than SMs: the lean decode kernel lets two sit beside its
      // three CTAs per SM (the Huginn shape, 220 CTAs: anchor-loop call 31.2 ->
      // 25.2 us; ouro8k batch 8, 256 CTAs: 45.2 -> 42.6 us; batch 16, 512 CTAs:
      // 77.2 -> 75.3 us).  With 128 CTAs, or 1024 (batch 32: 144.5 against
      // 147.1 us), the 72-register kernel is faster.
      const int coders = bhs + km_extra;
      if (coders > num_sms && coders <= 4 * num_sms) k = decode_kernel<D, GS, 0, PAGED, true>;
    }
  constexpr size_t merge_smem = NRES > 0 ? (size_t)D * D * sizeof(float) : 0;
  // Kernel attributes are per device: they are set, and the resident decode CTAs
  // per SM (registers and shared memory) found, on the first call made with each
  // device current.  Two threads racing on a first call both set the same values.
  static std::atomic<int> per_sm_dev[kMaxDevices];
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return e0;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int per_sm = per_sm_dev[dev].load(std::memory_order_acquire);
  if (per_sm == 0) {
    auto k0 = decode_kernel<D, GS, NRES, PAGED>;   // the lean variant is set up beside it
    // the stages and the kernel's own shared memory must fit one CTA's limit
    int optin = 0;
    e0 = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e0 != cudaSuccess) return e0;
    cudaFuncAttributes fa;
    e0 = cudaFuncGetAttributes(&fa, k0);
    if (e0 != cudaSuccess) return e0;
    if ((size_t)C::SMEM + fa.sharedSizeBytes > (size_t)optin) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k0, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if constexpr (NRES == 0) {   // both anchor-only decode kernels (same shared memory)
      e = cudaFuncSetAttribute(decode_kernel<D, GS, 0, PAGED, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(decode_kernel<D, GS, 0, PAGED, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               100);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(merge_kernel<D, (NRES > 0 ? 1 : 0), false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)merge_smem);
    if (e != cudaSuccess) return e;
    // All kernels of a call ask for the largest shared-memory carveout: the SM's
    // split between L1 and shared memory is fixed while CTAs are resident, so
    // a kernel that asks for another split waits for SMs to drain instead of
    // starting beside the kernel before it (its programmatic-dependent launch).
    e = cudaFuncSetAttribute(k0, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(qprep_kernel<D, GS, NRES>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(merge_kernel<D, (NRES > 0 ? 1 : 0), false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             100);
    if (e != cudaSuccess) return e;
    if constexpr (NRES == 0) {
      e = cudaFuncSetAttribute(merge_kernel<D, 0, true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k0, kThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorNotSupported;
    per_sm = occ < C::MINB ? occ : C::MINB;
    per_sm_dev[dev].store(per_sm, std::memory_order_release);
  }
  const int grid = num_sms * per_sm;
  if (grid > kMaxContrib) return cudaErrorNotSupported;   // merge_kernel's contributor table
  cudaError_t e = launch_dependent(qprep_kernel<D, GS, NRES>, dim3(bhs), dim3(kPrepThreads), 0, stream, a);
  if (e != cudaSuccess) return e;
  e = launch_dependent(k, dim3(grid), dim3(kThreads), (size_t)C::SMEM, stream, a);
  if (e != cudaSuccess) return e;
  return launch_dependent(km, dim3(bhs + km_extra), dim3(km_threads), km_smem, stream, a, grid);
}

}  // namespace
}  // namespace rq

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
  uint32_t* packs;       // [batch*H][NG][kPackWords]
  int pstride;
  int layer, group, batch, res0;   // res0: first residual plane this loop reads
  float qscale;                    // softmax_scale * log2(e)
};

// Chained calls that read 4 to 7 residual planes (rq_decode_chained.cu).
cudaError_t launch_decode_long_chain(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream);

namespace {

constexpr int kThreads = 256;
constexpr int kMaxCtasPerSm = 3;     // the workspace holds partials for this many CTAs per SM
constexpr int kMaxRows = RQ_MAX_DECODE_BATCH;   // batch rows one call may cover
constexpr int kMaxRes = 7;             // residual planes one call may read (chained, 8 loops)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFix = 32767.f;        // 16-bit fixed point: values in [-32767, 32767]
constexpr int kPackWords = 36;         // query pack per (row, head, group): anchor 16, residual 16, 4 scalars
constexpr int kPrepThreads = 256;
constexpr int kMergeThreads = 256;
constexpr int kMaxContrib = 512;       // decode CTAs one merge can combine (the grid is smaller)


__device__ __forceinline__ int dp4a_us(uint32_t a_u8, uint32_t b_s8, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8), "r"(b_s8), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a_u8, uint32_t b_u8, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8), "r"(b_u8), "r"(c));
  return d;
}
__device__ __forceinline__ int shl(int x, int s) { return (int)((uint32_t)x << s); }
// 16-bit fixed point value x = 256*hi + lo, hi in [-128, 127] (int8), lo in [0, 255]
__device__ __forceinline__ uint32_t fix_hi(int x) { return (uint32_t)(x >> 8) & 0xFFu; }
__device__ __forceinline__ uint32_t fix_lo(int x) { return (uint32_t)x & 0xFFu; }
__device__ __forceinline__ int to_fix(float x, float inv) {
  int v = __float2int_rn(x * inv);
  return max(-32767, min(32767, v));
}
__device__ __forceinline__ float2 meta2(const uint8_t* p) {   // (scale, offset)
  return e4m3x2_to_f32x2(*reinterpret_cast<const uint16_t*>(p));
}
__device__ __forceinline__ int clamp_len(int n, int nmax) { return n < 0 ? 0 : (n > nmax ? nmax : n); }

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
  static constexpr int NGP = NG <= 2 ? 2 : (NG <= 4 ? 4 : 8);   // groups padded to a power of two
  static constexpr int A_CODES = kTile * D / 2;
  static constexpr int R_CODES = kTile * D / 4;
  static constexpr int META = kTile * NG * 2;
  static constexpr int A_TILE = A_CODES + META;
  static constexpr int R_TILE = R_CODES + META + kTile * 2;
  static constexpr int SUB = 2 * A_TILE + 2 * NRES * R_TILE;      // one 64-token layout tile
  static constexpr int UT = 2;                                    // layout tiles per work unit
  static constexpr int UTOK = UT * kTile;                         // tokens per work unit
  static constexpr int STAGE = UT * SUB;
  static constexpr int STAGES = 2;
  // CTAs per SM: three (24 warps) while the registers allow it; the chained
  // variants with more residual planes keep two, or one from four planes up
  // (their two stages alone take most of the shared memory)
  static constexpr int MINB = NRES <= 1 ? 3 : (NRES <= 3 ? 2 : 1);
  static constexpr int PPT = UTOK * NGP / kThreads;               // (token, group) pairs per thread
  static constexpr int AW = GS / 8;              // 32-bit words of INT4 codes per (token, group)
  static constexpr int RW = GS / 16;             // 32-bit words of INT2 codes per (token, group)
  static constexpr int NITEM = NG * (1 + NRES);  // (kind, group) value-weight items per unit
  static constexpr int WQ = 2 * UTOK + 16;       // weight bytes per item: hi by token, lo by token, pad
  static constexpr int SMEM = STAGES * STAGE;
};

// Query packs of one (row, head): for each group, the 16-bit fixed-point query
// as int8 (hi, lo) parts laid out as the dp4a operands of the scoring, their
// scales and sums.  Words of pack (bh, group):
//   [4w + k], w < GS/8        anchor word w: k = 0 even-channel hi, 1 even lo,
//                             2 odd hi, 3 odd lo (channels 8w + 2i (+1), i = byte)
//   [16 + 8w + 2m + p]        residual word w, 2-bit field m: p = 0 hi, 1 lo
//                             (channels 16w + 4i + m, i = byte)
//   [32..35]                  sig_a, sum(q), sig_r, sum(R q) of the group (float bits)
template <int D, int GS, int NRES>
__global__ void __launch_bounds__(kPrepThreads) qprep_kernel(DecodeArgs a) {
  constexpr int NG = D / GS;
  constexpr int RPW = 16;                  // rows of R per warp (D / 8 <= 16; the rest padded)
  __shared__ __align__(16) float q_s[D];
  __shared__ float qr_s[D];
  __shared__ __align__(16) uint32_t img_s[NG * kPackWords];   // the packs of this (row, head)
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
  // stream: everything else read here (q) or written (the packs, which the
  // previous call's decode kernel may still read) waits for that kernel.  The
  // decode kernel is released at once: while the previous call drains, it
  // splits the work and starts its first cache copies.  What it reads before
  // its own wait (seq_lens, the cache) no kernel of this library writes while
  // released early: the kernels that write the cache (the append kernel, the
  // anchor-loop merge with the token append) release their dependents only when
  // they complete, and a caller's kernel does so too.
  pdl_launch_dependents();
  pdl_wait();
  if (tid < D) q_s[tid] = __bfloat162float(a.q[(size_t)bh * D + tid]) * a.qscale;
  for (int i = tid; i < NG * kPackWords; i += kPrepThreads) img_s[i] = 0u;
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
  // Each pack byte is written by the thread of its channel: thread k < D holds
  // channel k of q and of R q.  A group's GS channels sit in GS consecutive lanes
  // of one warp, so group maxima and sums are lane reductions.
  uint8_t* img = reinterpret_cast<uint8_t*>(img_s);
  if (tid < D) {
    const int k = tid, gi = k / GS, j = k % GS;
    const float x = q_s[k];
    float mx = fabsf(x), s1 = x;
#pragma unroll
    for (int off = GS / 2; off > 0; off >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    const int v = to_fix(x, mx > 0.f ? kFix / mx : 0.f);
    const int w = j >> 3, i = (j & 7) >> 1, odd = j & 1;
    uint8_t* wb = img + 4 * (gi * kPackWords + 4 * w + 2 * odd) + i;
    wb[0] = (uint8_t)fix_hi(v);
    wb[4] = (uint8_t)fix_lo(v);
    if (j == 0) {
      img_s[gi * kPackWords + 32] = __float_as_uint(mx / (kFix * 16.f));   // anchor sums carry 16
      img_s[gi * kPackWords + 33] = __float_as_uint(s1);
    }
  }
  if (NRES > 0 && tid < D) {
    const int k = tid, gi = k / GS, j = k % GS;
    const float x = qr_s[k];
    float mr = fabsf(x), s2 = x;
#pragma unroll
    for (int off = GS / 2; off > 0; off >>= 1) {
      mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, off));
      s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    }
    const int v = to_fix(x, mr > 0.f ? kFix / mr : 0.f);
    const int w = j >> 4, i = (j & 15) >> 2, m = j & 3;
    uint8_t* wb = img + 4 * (gi * kPackWords + 16 + 8 * w + 2 * m) + i;
    wb[0] = (uint8_t)fix_hi(v);
    wb[4] = (uint8_t)fix_lo(v);
    if (j == 0) {
      img_s[gi * kPackWords + 34] = __float_as_uint(mr / (kFix * 64.f));   // residual sums carry 64
      img_s[gi * kPackWords + 35] = __float_as_uint(s2);
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(a.packs + (size_t)bh * NG * kPackWords);
  const uint4* src = reinterpret_cast<const uint4*>(img_s);
  for (int i = tid; i < NG * kPackWords / 4; i += kPrepThreads) dst[i] = src[i];
}

// PAGED: the cache uses the block-table layout (tile addresses through the table).
template <int D, int GS, int NRES, bool PAGED>
__global__ void __launch_bounds__(kThreads, (Cfg<D, GS, NRES>::MINB)) decode_kernel(DecodeArgs a) {
  using C = Cfg<D, GS, NRES>;
  constexpr int NG = C::NG, NGP = C::NGP, AW = C::AW, RW = C::RW, STAGES = C::STAGES;
  constexpr int NITEM = C::NITEM, UTOK = C::UTOK, PPT = C::PPT, WQ = C::WQ;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[STAGES];
  __shared__ int pre_s[kMaxRows + 1];
  __shared__ int nt_s[kMaxRows + 1];        // work units (128-token) per row; then a sentinel
  __shared__ int sl_s[kMaxRows];
  // per-unit scratch; the first two are double-buffered by unit parity
  __shared__ float red_s[2][kThreads / 32];        // per-warp score maxima
  __shared__ uint32_t tmax_s[2][NITEM];            // max |value weight| per item, float bits
  // value weights of the unit in 16-bit fixed point, per item: the hi bytes indexed by token,
  // then the lo bytes.  V rows put four consecutive tokens of a channel in the bytes of a
  // masked code word, so one 32-bit load here is the matching dp4a operand.
  __shared__ __align__(16) uint8_t wq_s[NITEM][WQ];
  __shared__ float wsum_s[kThreads / 32][NITEM + 1];   // per-warp partials of off_s
  __shared__ float off_s[NITEM + 1];               // per-segment offset sums; [NITEM] = softmax sum

  pdl_launch_dependents();   // the merge kernel may start staging R
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
  Cursor pc = locate(u0);   // producer cursor (thread 0 only)
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
    for (int k = 0; k < ntile; ++k) {
      uint8_t* d = dst + k * C::SUB;
      const int tile = t0 + k;
      const uint8_t* blk = region;   // paged: this head's block of the tile's page
      if constexpr (PAGED) {
        const int page = max(checked_page(a.g, next_raw_s[k], a.status), 0);   // a bad entry reads page 0
        blk = a.base + (((int64_t)a.layer * a.g.G + a.group) * a.g.num_pages + page) * a.g.page_bytes +
              (int64_t)kvh * a.g.head_block;
      }
      auto src = [&](bool anchor, int j, int kv) {
        if constexpr (PAGED)   // same offsets as Geom::tile_offset, with the tile sizes as constants
          return blk + (anchor ? kv * C::A_TILE : 2 * C::A_TILE + (2 * j + kv) * C::R_TILE);
        else
          return region + (anchor ? a.g.anchor_plane(kv) : a.g.res_plane(j, kv)) +
                 (int64_t)tile * (anchor ? C::A_TILE : C::R_TILE);
      };
      bulk_g2s_hint(d, src(true, 0, 0), C::A_TILE, &full_bar[stage], pol);
      bulk_g2s_hint(d + C::A_TILE, src(true, 0, 1), C::A_TILE, &full_bar[stage], pol);
#pragma unroll
      for (int r = 0; r < NRES; ++r) {
        uint8_t* d0 = d + 2 * C::A_TILE + 2 * r * C::R_TILE;
        bulk_g2s_hint(d0, src(false, a.res0 + r, 0), C::R_TILE, &full_bar[stage], pol);
        bulk_g2s_hint(d0 + C::R_TILE, src(false, a.res0 + r, 1), C::R_TILE, &full_bar[stage], pol);
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
  for (int i = tid; i < 2 * NITEM; i += kThreads) (&tmax_s[0][0])[i] = 0u;
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

  // ---- per-thread state ----
  const int gi1 = tid % NGP;              // phase-1 group of this thread (same for every pair)
  const bool g_ok = gi1 < NG;
  // query packs: anchor [AW words][E.hi, E.lo, O.hi, O.lo], residual [RW words][m][hi, lo]
  uint32_t qa[AW][4];
  uint32_t qrp[RW][4][2];
  float sig_a = 0.f, sig_r = 0.f, qsum = 0.f, qrsum = 0.f;
  float acc = 0.f;          // phase-2 accumulator: (channel, anchor|residual)
  float m_run = -INFINITY;
  float off_part[1 + NRES]; // partial offset sums of this thread's group: anchor, residual planes
  float l_part = 0.f;       // partial softmax denominator (threads of group 0)
#pragma unroll
  for (int j = 0; j <= NRES; ++j) off_part[j] = 0.f;
  int cur_bh = -1;
  bool aborted = false;
  int fail_u = 0;

  const int p2_ch = tid < D ? tid : tid - D;
  const bool p2_anchor = tid < D;
  const bool p2_active = tid < (NRES > 0 ? 2 * D : D);

  auto flush = [&](int bh) {
    // finish the segment's partials: offset sums per item and the softmax denominator,
    // per warp, then over the warps in a fixed order (repeated calls give equal bits)
#pragma unroll
    for (int j = 0; j <= NRES; ++j) {
      float x = off_part[j];
      for (int off = NGP; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      if (lane < NGP && g_ok) wsum_s[warp][j * NG + gi1] = x;
    }
    {
      float x = l_part;
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
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
    if (p2_active) {
      const int gi = p2_ch / GS;
      float v = acc;
      if (p2_anchor) {
        v += off_s[gi];
      } else {
#pragma unroll
        for (int r = 0; r < NRES; ++r) v += off_s[(1 + r) * NG + gi];
      }
      part[2 + (p2_anchor ? 0 : D) + p2_ch] = v;
    }
  };

  auto begin_segment = [&](int bh) {
    // this thread's group's query packs (written by qprep_kernel; read through L2)
    const int gq = g_ok ? gi1 : 0;
    const uint4* pk = reinterpret_cast<const uint4*>(a.packs + ((size_t)bh * NG + gq) * kPackWords);
    uint32_t w[kPackWords];
#pragma unroll
    for (int i = 0; i < kPackWords / 4; ++i) {
      const uint4 v = __ldcg(pk + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int x = 0; x < AW; ++x)
#pragma unroll
      for (int k = 0; k < 4; ++k) qa[x][k] = w[4 * x + k];
#pragma unroll
    for (int x = 0; x < RW; ++x)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        qrp[x][m][0] = w[16 + 8 * x + 2 * m];
        qrp[x][m][1] = w[16 + 8 * x + 2 * m + 1];
      }
    sig_a = __uint_as_float(w[32]);
    qsum = __uint_as_float(w[33]);
    sig_r = __uint_as_float(w[34]);
    qrsum = __uint_as_float(w[35]);
    m_run = -INFINITY;
    l_part = 0.f;
#pragma unroll
    for (int j = 0; j <= NRES; ++j) off_part[j] = 0.f;
    acc = 0.f;
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

    // ---- phase 1: score of each token; a token's NGP groups sit in adjacent lanes ----
    float wmax = -INFINITY;
    float sc[PPT];            // scores of this thread's tokens (every lane of a token has it)
#pragma unroll
    for (int pp = 0; pp < PPT; ++pp) {
      const int tok = (tid + pp * kThreads) / NGP;
      const uint8_t* sub = st + (tok >> 6) * C::SUB;   // layout tile of this token
      const int row = tok & (kTile - 1);
      float score = 0.f;
      if (g_ok && !aborted && tok < n_valid) {
        const int gi = gi1;
        const uint8_t* AK = sub;
        // anchor: INT4 token-major; masks give the even / (16 x) odd channels as bytes
        uint32_t aw[4];
        if (AW == 4) {
          uint4 v = *reinterpret_cast<const uint4*>(AK + row * (D / 2) + gi * (GS / 2));
          aw[0] = v.x; aw[1] = v.y; aw[2] = v.z; aw[3] = v.w;
        } else {
          uint2 v = *reinterpret_cast<const uint2*>(AK + row * (D / 2) + gi * (GS / 2));
          aw[0] = v.x; aw[1] = v.y; aw[2] = 0u; aw[3] = 0u;
        }
        int eh = 0, el = 0, oh = 0, ol = 0;
#pragma unroll
        for (int w = 0; w < AW; ++w) {
          const uint32_t lo4 = aw[w] & 0x0F0F0F0Fu, hi4 = aw[w] & 0xF0F0F0F0u;
          eh = dp4a_us(lo4, qa[w][0], eh);
          el = dp4a_uu(lo4, qa[w][1], el);
          oh = dp4a_us(hi4, qa[w][2], oh);
          ol = dp4a_uu(hi4, qa[w][3], ol);
        }
        const int ta = shl(shl(eh, 8) + el, 4) + shl(oh, 8) + ol;     // 16 x sum(q_fix * code)
        const float2 ma = meta2(AK + C::A_CODES + row * NG * 2 + gi * 2);
        const float score_a = fmaf(ma.x, (float)ta * sig_a, ma.y * qsum);
        score = score_a;
        if (NRES > 0) {
          float cprod = 1.f, sres = 0.f;
#pragma unroll
          for (int r = 0; r < NRES; ++r) {
            const uint8_t* RK = sub + 2 * C::A_TILE + 2 * r * C::R_TILE;
            uint32_t rw[2];
            if (RW == 2) {
              uint2 v = *reinterpret_cast<const uint2*>(RK + row * (D / 4) + gi * (GS / 4));
              rw[0] = v.x; rw[1] = v.y;
            } else {
              rw[0] = *reinterpret_cast<const uint32_t*>(RK + row * (D / 4) + gi * (GS / 4));
              rw[1] = 0u;
            }
            int hm[4] = {0, 0, 0, 0}, lm[4] = {0, 0, 0, 0};
#pragma unroll
            for (int w = 0; w < RW; ++w)
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const uint32_t bm = rw[w] & (0x03030303u << (2 * m));
                hm[m] = dp4a_us(bm, qrp[w][m][0], hm[m]);
                lm[m] = dp4a_uu(bm, qrp[w][m][1], lm[m]);
              }
            const int tr = shl(shl(hm[0], 8) + lm[0], 6) + shl(shl(hm[1], 8) + lm[1], 4) +
                           shl(shl(hm[2], 8) + lm[2], 2) + (shl(hm[3], 8) + lm[3]);   // 64 x dot
            const float2 mr = meta2(RK + C::R_CODES + row * NG * 2 + gi * 2);
            const float cr = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(RK + C::R_CODES + C::META + row * 2));
            // chained: plane r weighs the product of the coefficients before it
            sres = fmaf(cprod, fmaf(mr.x, (float)tr * sig_r, mr.y * qrsum), sres);
            cprod *= cr;
          }
          score = fmaf(cprod, score_a, sres);
        }
      }
#pragma unroll
      for (int off = 1; off < NGP; off <<= 1) score += __shfl_xor_sync(0xffffffffu, score, off);
      if (tok >= n_valid) score = -INFINITY;
      sc[pp] = score;
      wmax = fmaxf(wmax, score);
    }
    for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
    if (lane == 0) red_s[buf][warp] = wmax;
    if (__syncthreads_or(aborted)) {                   // B1: per-warp score maxima are in red_s
      fail_u = u;
      aborted = true;
      if (tid == 0) atomicExch(&a.status[0], 1);
      break;
    }
    // every warp has finished the previous unit: its stage can be refilled
    if (tid == 0 && it >= 1 && u - 1 + STAGES < u1) issue((it - 1) % STAGES);

    float m_tile = red_s[buf][0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m_tile = fmaxf(m_tile, red_s[buf][w]);
    const float m_new = fmaxf(m_run, m_tile);
    const float alpha = ex2_fast(m_run - m_new);   // 0 on the first unit (m_run = -inf)
    m_run = m_new;

    // the maxima of the other parity were last read before B1: clear them for the next unit
    if (tid < NITEM) tmax_s[buf ^ 1][tid] = 0u;

    // ---- value weights of this thread's (token, group) pairs: p * coefficients * scale,
    //      and the offset terms p * coefficients * offset summed on the fly ----
    float wv[PPT][1 + NRES];
#pragma unroll
    for (int j = 0; j <= NRES; ++j) off_part[j] *= alpha;
#pragma unroll
    for (int pp = 0; pp < PPT; ++pp) {
      const int tok = (tid + pp * kThreads) / NGP;
      const float pt = ex2_fast(sc[pp] - m_new);       // 0 for masked tokens
      if (gi1 == 0) l_part = fmaf(l_part, pp == 0 ? alpha : 1.f, pt);
#pragma unroll
      for (int j = 0; j <= NRES; ++j) wv[pp][j] = 0.f;
      if (g_ok && tok < n_valid) {
        const uint8_t* sub = st + (tok >> 6) * C::SUB;
        const int row = tok & (kTile - 1);
        float cprod = pt;   // p times the coefficients of the planes before the current one
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const uint8_t* RV = sub + 2 * C::A_TILE + (2 * r + 1) * C::R_TILE;
          const float2 mv = meta2(RV + C::R_CODES + row * NG * 2 + gi1 * 2);
          wv[pp][1 + r] = cprod * mv.x;
          off_part[1 + r] = fmaf(cprod, mv.y, off_part[1 + r]);
          cprod *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(RV + C::R_CODES + C::META + row * 2));
        }
        const float2 ma = meta2(sub + C::A_TILE + C::A_CODES + row * NG * 2 + gi1 * 2);
        wv[pp][0] = cprod * ma.x;
        off_part[0] = fmaf(cprod, ma.y, off_part[0]);
      }
    }
    // per-item max |w|: lanes of one group, then one shared atomic per warp and item
    // (|w| >= 0 orders like its bit pattern)
#pragma unroll
    for (int j = 0; j <= NRES; ++j) {
      float mx = 0.f;
#pragma unroll
      for (int pp = 0; pp < PPT; ++pp) mx = fmaxf(mx, fabsf(wv[pp][j]));
      for (int off = NGP; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane < NGP && g_ok) atomicMax(&tmax_s[buf][j * NG + gi1], __float_as_uint(mx));
    }
    __syncthreads();                                   // B2: per-item maxima are final
    if (g_ok) {
#pragma unroll
      for (int j = 0; j <= NRES; ++j) {
        const float mx = __uint_as_float(tmax_s[buf][j * NG + gi1]);
        // any scale near kFix / mx works: the weights are clamped to the 16-bit
        // range and dequantized with mx / kFix
        const float inv = mx > 0.f ? __fdividef(kFix, mx) : 0.f;
        uint8_t* wq = wq_s[j * NG + gi1];
#pragma unroll
        for (int pp = 0; pp < PPT; ++pp) {
          const int tok = (tid + pp * kThreads) / NGP;
          const int v = to_fix(wv[pp][j], inv);
          wq[tok] = (uint8_t)fix_hi(v);
          wq[UTOK + tok] = (uint8_t)fix_lo(v);
        }
      }
    }
    __syncthreads();                                   // B3: weight operands are in wq_s

    // ---- phase 2: value accumulation, thread = (channel, anchor | residual) ----
    if (p2_active) {
      const int gi = p2_ch / GS;
      float add = 0.f;
      if (p2_anchor) {
        const uint8_t* wq = wq_s[gi];
        int eh = 0, el = 0, oh = 0, ol = 0;
#pragma unroll
        for (int sb = 0; sb < C::UT; ++sb) {
          const uint4* row = reinterpret_cast<const uint4*>(st + sb * C::SUB + C::A_TILE + p2_ch * (kTile / 2));
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint4 x4 = row[h2];
            const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              // code words w, w+1 hold tokens 8w .. 8w+15; the low nibbles of word w are
              // tokens 8w .. 8w+3, the high nibbles 8w+4 .. 8w+7
              const int w = sb * 8 + h2 * 4 + q2 * 2;
              const uint4 wh = *reinterpret_cast<const uint4*>(wq + 8 * w);
              const uint4 wl = *reinterpret_cast<const uint4*>(wq + UTOK + 8 * w);
              const uint32_t a0 = xs[2 * q2], a1 = xs[2 * q2 + 1];
              eh = dp4a_us(a0 & 0x0F0F0F0Fu, wh.x, eh);
              el = dp4a_uu(a0 & 0x0F0F0F0Fu, wl.x, el);
              oh = dp4a_us(a0 & 0xF0F0F0F0u, wh.y, oh);
              ol = dp4a_uu(a0 & 0xF0F0F0F0u, wl.y, ol);
              eh = dp4a_us(a1 & 0x0F0F0F0Fu, wh.z, eh);
              el = dp4a_uu(a1 & 0x0F0F0F0Fu, wl.z, el);
              oh = dp4a_us(a1 & 0xF0F0F0F0u, wh.w, oh);
              ol = dp4a_uu(a1 & 0xF0F0F0F0u, wl.w, ol);
            }
          }
        }
        const int t = shl(shl(eh, 8) + el, 4) + shl(oh, 8) + ol;        // 16 x sum(w_fix * code)
        add = (float)t * (__uint_as_float(tmax_s[buf][gi]) * (1.f / (16.f * kFix)));
      } else {
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const int item = (1 + r) * NG + gi;
          const uint8_t* wq = wq_s[item];
          int hm[4] = {0, 0, 0, 0}, lm[4] = {0, 0, 0, 0};
#pragma unroll
          for (int sb = 0; sb < C::UT; ++sb) {
            const uint4 x4 = *reinterpret_cast<const uint4*>(st + sb * C::SUB + 2 * C::A_TILE +
                                                             (2 * r + 1) * C::R_TILE + p2_ch * (kTile / 4));
            const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // word j: mask 3 << 2m leaves tokens 16j + 4m .. 16j + 4m + 3
              const int t0 = sb * kTile + 16 * j;
              const uint4 wh = *reinterpret_cast<const uint4*>(wq + t0);
              const uint4 wl = *reinterpret_cast<const uint4*>(wq + UTOK + t0);
              const uint32_t b0 = xs[j] & 0x03030303u, b1 = xs[j] & 0x0C0C0C0Cu;
              const uint32_t b2 = xs[j] & 0x30303030u, b3 = xs[j] & 0xC0C0C0C0u;
              hm[0] = dp4a_us(b0, wh.x, hm[0]); lm[0] = dp4a_uu(b0, wl.x, lm[0]);
              hm[1] = dp4a_us(b1, wh.y, hm[1]); lm[1] = dp4a_uu(b1, wl.y, lm[1]);
              hm[2] = dp4a_us(b2, wh.z, hm[2]); lm[2] = dp4a_uu(b2, wl.z, lm[2]);
              hm[3] = dp4a_us(b3, wh.w, hm[3]); lm[3] = dp4a_uu(b3, wl.w, lm[3]);
            }
          }
          const int t = shl(shl(hm[0], 8) + lm[0], 6) + shl(shl(hm[1], 8) + lm[1], 4) +
                        shl(shl(hm[2], 8) + lm[2], 2) + (shl(hm[3], 8) + lm[3]);   // 64 x sum
          add = fmaf((float)t, __uint_as_float(tmax_s[buf][item]) * (1.f / (64.f * kFix)), add);
        }
      }
      acc = fmaf(acc, alpha, add);
    }
    // no barrier here: the next unit writes wq_s only after its B2 and clears this
    // parity's maxima only after its B1, and its stage is refilled after the next B1
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
}

// Combines the partial softmax states of (row, head) blockIdx.x: the CTAs that
// held its units are recomputed from seq_lens with the decode kernel's split.
// APPEND (anchor-loop call only): the grid has two CTAs per (row, head); they
// also compress the current token's K (first CTA, which also merges) and V
// (second CTA) into the cache at position seq_lens[row] (rq_token_append.cuh).
// They run 128 threads of at most 32 registers, small enough to sit beside the
// decode kernel's CTAs and do that work while those stream.
template <int D, int NRES, bool APPEND>
__global__ void __launch_bounds__(APPEND ? kAppendThreads : kMergeThreads, APPEND ? 16 : 0)
    merge_kernel(DecodeArgs a, int Cn) {
  static_assert(!APPEND || NRES == 0, "append runs in the anchor-loop merge");
  constexpr int NT = APPEND ? kAppendThreads : kMergeThreads;
  static_assert(NRES == 0 ? NT >= D : NT >= 2 * D, "a thread per accumulator element");
  extern __shared__ __align__(16) float R_s[];   // [D][D] when NRES > 0; the append's scratch with APPEND
  __shared__ float w_s[kMaxContrib];
  __shared__ float l_s[kMaxContrib];
  __shared__ float va_s[D];
  __shared__ float vr_s[D];
  __shared__ float rt_s[D];
  __shared__ float redf_s[NT / 32];
  __shared__ int redi_s[2][NT / 32];
  __shared__ float ml_s[2];
  __shared__ uint64_t r_bar;
  constexpr int UTOK = 2 * kTile;
  // the next call's prep may start loading R (it waits for this kernel); the
  // appending variant writes the cache, so its dependents wait for it to finish
  if constexpr (!APPEND) pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.g.Hq, B = a.batch, Hkv = a.g.H;   // merge CTAs: one per (row, query head)
  // APPEND: CTAs [0, B*Hq) merge, the first query head of each KV head also coding
  // the token's K; CTAs [B*Hq, B*Hq + B*Hkv) code the V of one (row, KV head)
  const bool v_cta = APPEND && (int)blockIdx.x >= B * H;
  int bh, b, h, kvh;
  if (v_cta) {
    const int r = blockIdx.x - B * H;
    b = r / Hkv;
    kvh = r - b * Hkv;
    h = kvh * a.g.qpk;
    bh = b * H + h;
  } else {
    bh = blockIdx.x;
    b = bh / H;
    h = bh - b * H;
    kvh = h / a.g.qpk;
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
  // current token's score (base 2)
  float sc = 0.f;
  for (int k = tid; k < D; k += NT)
    sc += __bfloat162float(a.q[(size_t)bh * D + k]) * a.qscale *
          __bfloat162float(a.k_cur[(size_t)kvbh * D + k]);
  // units before this row and in total (same clamping and unit size as the decode kernel)
  int before = 0, total = 0;
  for (int r = tid; r < B; r += NT) {
    const int nt = (clamp_len(a.seq_lens[r], a.g.Nmax) + UTOK - 1) / UTOK;
    total += H * nt;
    if (r < b) before += H * nt;
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
    for (int k = tid; k < D; k += NT)
      a.out[(size_t)bh * D + k] = __bfloat162float(a.v_cur[(size_t)kvbh * D + k]);
    if constexpr (APPEND)
      if (app_ok)
        token_append_store<D>(a.g, const_cast<uint8_t*>(a.base), a.layer, a.group, b, kvh, 0, app_pos, app_page,
                              app_smem);
    return;
  }
  const Split split{U / Cn, U % Cn};
  const int s0 = pre + h * ntb, s1 = s0 + ntb;
  const int c_lo = split.owner(s0), c_hi = split.owner(s1 - 1);
  const int nc = min(c_hi - c_lo + 1, kMaxContrib);

  pdl_wait();   // every partial of the decode kernel is written and visible
  if constexpr (APPEND)   // no kernel before this one is running: the new slot can be written
    if (app_ok)
      token_append_store<D>(a.g, const_cast<uint8_t*>(a.base), a.layer, a.group, b, kvh, 0, app_pos, app_page,
                            app_smem);

  // this thread's element of the first contributors' accumulators, loaded while
  // warp 0 reads the (m, l) pairs
  constexpr int PF = 8;
  const bool acc_thread = tid < (NRES > 0 ? 2 * D : D);   // NT covers them (static_assert above)
  const float* pc = a.partials + (size_t)(c_lo + bh) * a.pstride + 2 + tid;
  float xa[PF];
#pragma unroll
  for (int k = 0; k < PF; ++k) xa[k] = (acc_thread && k < nc) ? __ldcg(pc + (size_t)k * a.pstride) : 0.f;
  if (warp == 0) {
    // (m, l) of each contributor, read once: m parked in w_s, l in l_s
    float M = s_cur;
    for (int i = lane; i < nc; i += 32) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.partials + (size_t)(c_lo + i + bh) * a.pstride));
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
  const float M = ml_s[0], L = ml_s[1];
  // thread = (channel, anchor | residual accumulator)
  if (acc_thread) {
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < PF; ++k)
      if (k < nc) v = fmaf(w_s[k], xa[k], v);
    for (int i = PF; i < nc; ++i) v = fmaf(w_s[i], __ldcg(pc + (size_t)i * a.pstride), v);
    if (tid < D) va_s[tid] = fmaf(exp2f(s_cur - M), __bfloat162float(a.v_cur[(size_t)kvbh * D + tid]), v);
    else vr_s[tid - D] = v;
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
        t0 = fmaf(rc[(k + 0) * D], vr[k + 0], t0);
        t1 = fmaf(rc[(k + 1) * D], vr[k + 1], t1);
        t2 = fmaf(rc[(k + 2) * D], vr[k + 2], t2);
        t3 = fmaf(rc[(k + 3) * D], vr[k + 3], t3);
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
  size_t km_smem = NRES > 0 ? (size_t)D * D * sizeof(float) : 0;
  if (a.g.mode & RQ_MODE_HADAMARD) km_smem = 0;   // no R to stage
  int km_threads = kMergeThreads, km_extra = 0;
  if constexpr (NRES == 0)
    if (a.kv_all) {
      km = merge_kernel<D, 0, true>;
      km_smem = TokenAppendSmem::bytes(a.g.P);
      km_threads = kAppendThreads;
      km_extra = a.batch * a.g.H;   // the V-coding CTAs, one per (row, KV head)
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
    // the stages and the kernel's own shared memory must fit one CTA's limit
    int optin = 0;
    e0 = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e0 != cudaSuccess) return e0;
    cudaFuncAttributes fa;
    e0 = cudaFuncGetAttributes(&fa, k);
    if (e0 != cudaSuccess) return e0;
    if ((size_t)C::SMEM + fa.sharedSizeBytes > (size_t)optin) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(merge_kernel<D, (NRES > 0 ? 1 : 0), false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)merge_smem);
    if (e != cudaSuccess) return e;
    // All kernels of a call ask for the largest shared-memory carveout: the SM's
    // split between L1 and shared memory is fixed while CTAs are resident, so
    // a kernel that asks for another split waits for SMs to drain instead of
    // starting beside the kernel before it (its programmatic-dependent launch).
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
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
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorNotSupported;
    per_sm = occ < C::MINB ? occ : C::MINB;
    per_sm_dev[dev].store(per_sm, std::memory_order_release);
  }
  const int grid = num_sms * per_sm;
  if (grid > kMaxContrib) return cudaErrorNotSupported;   // merge_kernel's contributor table
  const int bhs = a.batch * a.g.Hq;   // (row, query head) pairs
  cudaError_t e = launch_dependent(qprep_kernel<D, GS, NRES>, dim3(bhs), dim3(kPrepThreads), 0, stream, a);
  if (e != cudaSuccess) return e;
  e = launch_dependent(k, dim3(grid), dim3(kThreads), (size_t)C::SMEM, stream, a);
  if (e != cudaSuccess) return e;
  return launch_dependent(km, dim3(bhs + km_extra), dim3(km_threads), km_smem, stream, a, grid);
}

}  // namespace
}  // namespace rq

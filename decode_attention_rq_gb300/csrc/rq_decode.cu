// rq_decode_attention: split-K decode attention over the compressed cache.
//
// The explainer "ResidualQuant stores looped-Transformer KV caches as 2-bit
// residuals" (paragraph on the custom attention kernel and the one on shared
// versus chained anchors) fixes what the kernel must do: rebuild each loop's
// K/V as c * anchor + residual tile by tile in on-chip memory, never writing
// the rebuilt tensor back; a shared anchor needs two plane reads per key, a
// chained one reads every residual between the loop and the anchor.
//
// GB300 design
//   * Work units are (row, head, 64-token tile).  A fixed grid of
//     num_SMs x kCtasPerSm CTAs takes equal contiguous ranges of the flattened
//     unit list (ranges cross (row, head) boundaries), so every SM streams
//     the same number of tiles whatever the batch and lengths.
//   * A tile's plane slices (anchor K/V, the residual K/V planes this loop
//     reads) are contiguous and 16-byte aligned: one thread issues 1-D TMA
//     bulk copies into a shared-memory ring tracked by mbarriers (bounded
//     waits); all other threads only compute.
//   * Scores use the rotated query: q.(c a_hat + R^T r_hat) = c (q.a_hat) +
//     (R q).r_hat.  R is applied to q once per (row, head) segment; the value
//     side accumulates the anchor part and the rotated residual part apart,
//     and R^T is applied once, at the merge.
//   * Per group, q.x_hat = s * sum(q * code) + o * sum(q), and the value side
//     keeps the offsets as one scalar per (tile, group): the work per code is
//     one multiply-add against a small integer.
//   * That multiply-add runs on the integer dot-product unit: the query (per
//     group) and the softmax-times-scale weights (per tile and group) are
//     taken to 16-bit fixed point as two int8 parts; dp4a sums 4 code x part
//     products exactly.  Byte masks put the codes straight into dp4a operands:
//     K rows are token-major (4 codes of one token per operand), V rows are
//     channel-major (4 tokens of one channel per operand), so no shifts are
//     needed.  The masks and the dot products run on separate pipes of the
//     SM and overlap.
//   * Online softmax in base 2 (scale * log2(e) folded into q).  Each CTA
//     writes one partial (m, l, acc_anchor, acc_residual) per segment; the
//     last CTA to finish a (row, head) -- an atomic counter, no spinning --
//     merges the partials, adds the current BF16 token, applies R^T and
//     writes the output.
#include <cuda_fp8.h>

#include "rq_internal.cuh"

namespace rq {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 2;
constexpr int kMaxRows = 256;          // batch rows one call may cover
constexpr int kMaxRes = 3;             // residual planes one call may read (chained, 4 loops)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFix = 32767.f;        // 16-bit fixed point: values in [-32767, 32767]

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
  int32_t* counters;     // [batch * H]
  float* partials;       // [(C + batch*H)][pstride]
  int pstride;
  int layer, group, batch, res0;   // res0: first residual plane this loop reads
  float qscale;                    // softmax_scale * log2(e)
};

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

// flattened unit u -> CTA that owns it, for ranges [floor(cU/C), floor((c+1)U/C))
__device__ __forceinline__ int cta_of(long long u, long long U, int C) {
  return (int)(((u + 1) * C - 1) / U);
}
// CTA c's range intersects [s0, s1) (ranges are empty when units < CTAs)
__device__ __forceinline__ bool contributes(int c, long long s0, long long s1, long long U, int C) {
  long long r0 = (long long)c * U / C, r1 = (long long)(c + 1) * U / C;
  return (r0 > s0 ? r0 : s0) < (r1 < s1 ? r1 : s1);
}

template <int D, int GS, int NRES>
struct Cfg {
  static constexpr int NG = D / GS;
  static constexpr int NGP = NG <= 2 ? 2 : (NG <= 4 ? 4 : 8);   // groups padded to a power of two
  static constexpr int A_CODES = kTile * D / 2;
  static constexpr int R_CODES = kTile * D / 4;
  static constexpr int META = kTile * NG * 2;
  static constexpr int A_TILE = A_CODES + META;
  static constexpr int R_TILE = R_CODES + META + kTile * 2;
  static constexpr int STAGES = NRES >= 2 ? 3 : 4;
  static constexpr int STAGE = 2 * A_TILE + 2 * NRES * R_TILE;
  static constexpr int PPT = kTile * NGP / kThreads;        // (token, group) pairs per thread
  static constexpr int AW = GS / 8;              // 32-bit words of INT4 codes per (token, group)
  static constexpr int RW = GS / 16;             // 32-bit words of INT2 codes per (token, group)
  static constexpr int NITEM = NG * (1 + NRES);  // (kind, group) value-weight items per tile
  static constexpr int SMEM = STAGES * STAGE;
};

template <int D, int GS, int NRES>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(DecodeArgs a) {
  using C = Cfg<D, GS, NRES>;
  constexpr int NG = C::NG, NGP = C::NGP, AW = C::AW, RW = C::RW, STAGES = C::STAGES;
  constexpr int NITEM = C::NITEM;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[STAGES];
  __shared__ int pre_s[kMaxRows + 1];
  __shared__ int nt_s[kMaxRows];
  __shared__ __align__(16) float q_s[D];
  __shared__ __align__(16) float qr_s[D];
  // per-tile scratch, double-buffered by tile parity
  __shared__ float s_s[2][kTile];                  // token scores (base-2 logits)
  __shared__ float red_s[2][kThreads / 32];        // per-warp score maxima
  __shared__ float tau_s[2][NITEM], off_s[2][NITEM];
  // dp4a operands of the value weights, one 32-bit word per lane of the item's warp:
  // anchor item: [8 words][E.hi, E.lo, O.hi, O.lo]; residual item: [4 words][mask m][hi, lo]
  __shared__ __align__(16) uint32_t pack_s[2][NITEM][32];
  __shared__ float mrg_s[8];
  __shared__ float m_sh, l_sh;
  __shared__ int flag_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.g.H, B = a.batch;
  const int Cn = gridDim.x, cta = blockIdx.x;

  // ---- per-row tile counts and prefix over (row, head) ----
  for (int b = tid; b < B; b += kThreads) {
    int n = a.seq_lens[b];
    n = n < 0 ? 0 : (n > a.g.Nmax ? a.g.Nmax : n);
    nt_s[b] = (n + kTile - 1) / kTile;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      pre_s[b] = acc;
      acc += H * nt_s[b];
    }
    pre_s[B] = acc;
  }
  __syncthreads();
  const long long U = pre_s[B];

  // ---- (row, head) pairs with an empty cache: the output is the current V ----
  for (int bh = cta; bh < B * H; bh += Cn) {
    if (nt_s[bh / H] != 0) continue;
    for (int k = tid; k < D; k += kThreads)
      a.out[(size_t)bh * D + k] = __bfloat162float(a.v_cur[(size_t)bh * D + k]);
  }
  if (U == 0) return;
  const long long u0 = (long long)cta * U / Cn, u1 = (long long)(cta + 1) * U / Cn;
  if (u0 >= u1) return;

  auto locate = [&](long long u, int* bh, int* tile) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {   // last row b with pre_s[b] <= u (rows with no tiles are skipped)
      int mid = (lo + hi + 1) >> 1;
      if (pre_s[mid] <= u) lo = mid; else hi = mid - 1;
    }
    int rem = (int)(u - pre_s[lo]);
    *bh = lo * H + rem / nt_s[lo];
    *tile = rem % nt_s[lo];
  };
  auto issue = [&](long long u, int stage) {
    int bh, tile;
    locate(u, &bh, &tile);
    const uint8_t* region = a.base + a.g.region_offset(a.layer, a.group, bh / H, bh % H);
    uint8_t* dst = smem + stage * C::STAGE;
    mbar_arrive_expect_tx(&full_bar[stage], C::STAGE);
    bulk_g2s(dst, region + a.g.anchor_plane(0) + (int64_t)tile * C::A_TILE, C::A_TILE, &full_bar[stage]);
    bulk_g2s(dst + C::A_TILE, region + a.g.anchor_plane(1) + (int64_t)tile * C::A_TILE, C::A_TILE,
             &full_bar[stage]);
#pragma unroll
    for (int r = 0; r < NRES; ++r) {
      uint8_t* d0 = dst + 2 * C::A_TILE + 2 * r * C::R_TILE;
      bulk_g2s(d0, region + a.g.res_plane(a.res0 + r, 0) + (int64_t)tile * C::R_TILE, C::R_TILE,
               &full_bar[stage]);
      bulk_g2s(d0 + C::R_TILE, region + a.g.res_plane(a.res0 + r, 1) + (int64_t)tile * C::R_TILE,
               C::R_TILE, &full_bar[stage]);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&full_bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < STAGES && u0 + s < u1; ++s) issue(u0 + s, s);

  // ---- per-thread state ----
  const int gi1 = tid % NGP;              // phase-1 group of this thread (same for every pair)
  const bool g_ok = gi1 < NG;
  // query packs: anchor [AW words][E.hi, E.lo, O.hi, O.lo], residual [RW words][m][hi, lo]
  uint32_t qa[AW][4];
  uint32_t qrp[RW][4][2];
  float sig_a = 0.f, sig_r = 0.f, qsum = 0.f, qrsum = 0.f;
  float acc = 0.f;          // phase-2 accumulator: (channel, anchor|residual)
  float m_run = -INFINITY, l_run = 0.f;   // l_run is kept by thread 0
  int cur_bh = -1;
  bool aborted = false;
  long long fail_u = 0;

  const int p2_ch = tid < D ? tid : tid - D;
  const bool p2_anchor = tid < D;
  const bool p2_active = tid < (NRES > 0 ? 2 * D : D);

  auto flush = [&](int bh) {
    // write this CTA's partial for bh, then the last CTA merges
    float* part = a.partials + (size_t)(cta + bh) * a.pstride;
    if (tid == 0) {
      part[0] = m_run;
      part[1] = l_run;
    }
    if (p2_active) part[2 + (p2_anchor ? 0 : D) + p2_ch] = acc;
    __threadfence();
    __syncthreads();
    const int b = bh / H, h = bh % H;
    const long long s0 = pre_s[b] + (long long)h * nt_s[b];
    const long long s1 = s0 + nt_s[b];
    const int c_lo = cta_of(s0, U, Cn), c_hi = cta_of(s1 - 1, U, Cn);
    if (tid == 0) {
      int needed = 0;
      for (int c = c_lo; c <= c_hi; ++c) needed += contributes(c, s0, s1, U, Cn);
      int prev = atomicAdd(&a.counters[bh], 1);
      flag_s = (prev == needed - 1);
    }
    __syncthreads();
    if (!flag_s) return;
    __threadfence();
    // ---- merge (this CTA is the last one for bh) ----
    float sc = 0.f;
    for (int k = tid; k < D; k += kThreads) sc += q_s[k] * __bfloat162float(a.k_cur[(size_t)bh * D + k]);
    for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
    if (lane == 0) mrg_s[warp] = sc;
    __syncthreads();
    if (tid == 0) {
      float s_cur = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) s_cur += mrg_s[w];
      float M = s_cur;
      for (int c = c_lo; c <= c_hi; ++c)
        if (contributes(c, s0, s1, U, Cn)) M = fmaxf(M, __ldcg(a.partials + (size_t)(c + bh) * a.pstride));
      float L = exp2f(s_cur - M);
      for (int c = c_lo; c <= c_hi; ++c) {
        if (!contributes(c, s0, s1, U, Cn)) continue;
        const float* pc = a.partials + (size_t)(c + bh) * a.pstride;
        L += __ldcg(pc + 1) * exp2f(__ldcg(pc) - M);
      }
      m_sh = M;
      l_sh = L;
      mrg_s[0] = s_cur;
    }
    __syncthreads();
    const float M = m_sh, L = l_sh, s_cur = mrg_s[0];
    if (tid < D) {
      float va = 0.f, vr = 0.f;
      for (int c = c_lo; c <= c_hi; ++c) {
        if (!contributes(c, s0, s1, U, Cn)) continue;
        const float* pc = a.partials + (size_t)(c + bh) * a.pstride;
        float w = exp2f(__ldcg(pc) - M);
        va = fmaf(w, __ldcg(pc + 2 + tid), va);
        if (NRES > 0) vr = fmaf(w, __ldcg(pc + 2 + D + tid), vr);
      }
      va = fmaf(exp2f(s_cur - M), __bfloat162float(a.v_cur[(size_t)bh * D + tid]), va);
      if (NRES > 0) qr_s[tid] = vr;
      q_s[tid] = va;
    }
    __syncthreads();
    if (tid < D) {
      float o = q_s[tid];
      if (NRES > 0) {
        float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;   // (R^T acc_r)[tid], loads coalesced over tid
#pragma unroll 4
        for (int k = 0; k < D; k += 4) {
          t0 = fmaf(__ldg(a.R + (size_t)(k + 0) * D + tid), qr_s[k + 0], t0);
          t1 = fmaf(__ldg(a.R + (size_t)(k + 1) * D + tid), qr_s[k + 1], t1);
          t2 = fmaf(__ldg(a.R + (size_t)(k + 2) * D + tid), qr_s[k + 2], t2);
          t3 = fmaf(__ldg(a.R + (size_t)(k + 3) * D + tid), qr_s[k + 3], t3);
        }
        o += (t0 + t1) + (t2 + t3);
      }
      a.out[(size_t)bh * D + tid] = o / L;
    }
    if (tid == 0) a.counters[bh] = 0;
    __syncthreads();
  };

  auto begin_segment = [&](int bh) {
    for (int k = tid; k < D; k += kThreads) q_s[k] = __bfloat162float(a.q[(size_t)bh * D + k]) * a.qscale;
    __syncthreads();
    if (NRES > 0) {
      // q' = R q: warp w takes rows w, w+8, ...; one coalesced float4 per lane
      for (int i = warp; i < D; i += kThreads / 32) {
        float t = 0.f;
        if (lane < D / 4) {
          float4 r = __ldg(reinterpret_cast<const float4*>(a.R + (size_t)i * D) + lane);
          float4 qv = *reinterpret_cast<const float4*>(&q_s[4 * lane]);
          t = r.x * qv.x + r.y * qv.y + r.z * qv.z + r.w * qv.w;
        }
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (lane == 0) qr_s[i] = t;
      }
      __syncthreads();
    }
    // fixed-point packs of this thread's phase-1 group
    const int gq = g_ok ? gi1 : 0;
    {
      const float* qg = q_s + gq * GS;
      float mx = 0.f, s1 = 0.f;
#pragma unroll
      for (int k = 0; k < GS; ++k) { mx = fmaxf(mx, fabsf(qg[k])); s1 += qg[k]; }
      const float inv = mx > 0.f ? kFix / mx : 0.f;
      sig_a = mx / (kFix * 16.f);              // anchor sums carry a factor 16
      qsum = s1;
#pragma unroll
      for (int w = 0; w < AW; ++w) {
        uint32_t eh = 0, el = 0, oh = 0, ol = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          int ve = to_fix(qg[8 * w + 2 * i], inv), vo = to_fix(qg[8 * w + 2 * i + 1], inv);
          eh |= fix_hi(ve) << (8 * i); el |= fix_lo(ve) << (8 * i);
          oh |= fix_hi(vo) << (8 * i); ol |= fix_lo(vo) << (8 * i);
        }
        qa[w][0] = eh; qa[w][1] = el; qa[w][2] = oh; qa[w][3] = ol;
      }
    }
    if (NRES > 0) {
      const float* rg = qr_s + gq * GS;
      float mr = 0.f, s2 = 0.f;
#pragma unroll
      for (int k = 0; k < GS; ++k) { mr = fmaxf(mr, fabsf(rg[k])); s2 += rg[k]; }
      const float invr = mr > 0.f ? kFix / mr : 0.f;
      sig_r = mr / (kFix * 64.f);            // residual sums carry a factor 64
      qrsum = s2;
#pragma unroll
      for (int w = 0; w < RW; ++w)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint32_t hh = 0, ll = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            int v = to_fix(rg[16 * w + 4 * i + m], invr);
            hh |= fix_hi(v) << (8 * i); ll |= fix_lo(v) << (8 * i);
          }
          qrp[w][m][0] = hh; qrp[w][m][1] = ll;
        }
    }
    m_run = -INFINITY;
    l_run = 0.f;
    acc = 0.f;
    cur_bh = bh;
    __syncthreads();   // q_s / qr_s may be rewritten by the next merge only after all packs are read
  };

  for (long long u = u0; u < u1; ++u) {
    const int it = (int)(u - u0), stage = it % STAGES, buf = it & 1;
    int bh, tile;
    locate(u, &bh, &tile);
    if (bh != cur_bh) {
      if (cur_bh >= 0) flush(cur_bh);
      begin_segment(bh);
    }
    const int n_valid = min(kTile, a.seq_lens[bh / H] - tile * kTile);

    if (!mbar_wait_bounded(&full_bar[stage], (uint32_t)((it / STAGES) & 1))) aborted = true;

    const uint8_t* st = smem + stage * C::STAGE;
    const uint8_t* AK = st;
    const uint8_t* AV = st + C::A_TILE;
    const uint8_t* RES = st + 2 * C::A_TILE;     // plane r: K at RES + 2r*R_TILE, V right after

    // ---- phase 1: score of each token; a token's NGP groups sit in adjacent lanes ----
    float wmax = -INFINITY;
#pragma unroll
    for (int pp = 0; pp < C::PPT; ++pp) {
      const int tok = (tid + pp * kThreads) / NGP;
      float score = 0.f;
      if (g_ok && !aborted) {
        const int gi = gi1;
        // anchor: INT4 token-major; masks give the even / (16 x) odd channels as bytes
        uint32_t aw[4];
        if (AW == 4) {
          uint4 v = *reinterpret_cast<const uint4*>(AK + tok * (D / 2) + gi * (GS / 2));
          aw[0] = v.x; aw[1] = v.y; aw[2] = v.z; aw[3] = v.w;
        } else {
          uint2 v = *reinterpret_cast<const uint2*>(AK + tok * (D / 2) + gi * (GS / 2));
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
        const float2 ma = meta2(AK + C::A_CODES + tok * NG * 2 + gi * 2);
        const float score_a = fmaf(ma.x, (float)ta * sig_a, ma.y * qsum);
        score = score_a;
        if (NRES > 0) {
          float cprod = 1.f, sres = 0.f;
#pragma unroll
          for (int r = 0; r < NRES; ++r) {
            const uint8_t* RK = RES + 2 * r * C::R_TILE;
            uint32_t rw[2];
            if (RW == 2) {
              uint2 v = *reinterpret_cast<const uint2*>(RK + tok * (D / 4) + gi * (GS / 4));
              rw[0] = v.x; rw[1] = v.y;
            } else {
              rw[0] = *reinterpret_cast<const uint32_t*>(RK + tok * (D / 4) + gi * (GS / 4));
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
            const float2 mr = meta2(RK + C::R_CODES + tok * NG * 2 + gi * 2);
            const float cr = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(RK + C::R_CODES + C::META + tok * 2));
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
      if (gi1 == 0) s_s[buf][tok] = score;
      wmax = fmaxf(wmax, score);
    }
    for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
    if (lane == 0) red_s[buf][warp] = wmax;
    if (__syncthreads_or(aborted)) {                   // B1: scores of the tile are in s_s
      fail_u = u;
      aborted = true;
      if (tid == 0) atomicExch(&a.status[0], 1);
      break;
    }
    // every warp has finished the previous tile: its stage can be refilled
    if (tid == 0 && it >= 1 && u - 1 + STAGES < u1) issue(u - 1 + STAGES, (it - 1) % STAGES);

    float m_tile = red_s[buf][0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m_tile = fmaxf(m_tile, red_s[buf][w]);
    const float m_new = fmaxf(m_run, m_tile);
    const float alpha = exp2f(m_run - m_new);   // 0 on the first tile (m_run = -inf)
    m_run = m_new;

    // ---- value weights: warp w takes items w, w+8, ... (item = (kind, group)) ----
    for (int item = warp; item < NITEM; item += kThreads / 32) {
      const int r = item / NG, gi = item % NG;      // r = 0 anchor, r >= 1 residual plane r-1
      float wv[2], ov[2];
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int tok = lane + 32 * hlf;
        const float pt = exp2f(s_s[buf][tok] - m_new);   // 0 for masked tokens (-inf)
        float w = 0.f, o = 0.f;
        if (tok < n_valid) {
          float cprod = 1.f;   // product of the coefficients of the planes before this one
          const int upto = r == 0 ? NRES : r - 1;
#pragma unroll
          for (int k = 0; k < NRES; ++k)
            if (k < upto)
              cprod *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(
                  RES + (2 * k + 1) * C::R_TILE + C::R_CODES + C::META + tok * 2));
          const uint8_t* mp = r == 0 ? AV + C::A_CODES : RES + (2 * (r - 1) + 1) * C::R_TILE + C::R_CODES;
          const float2 mv = meta2(mp + tok * NG * 2 + gi * 2);
          w = pt * cprod * mv.x;
          o = pt * cprod * mv.y;
        }
        wv[hlf] = w;
        ov[hlf] = o;
        if (item == 0) {   // the warp of item 0 also sums p for the softmax denominator
          float ps = pt;
          for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
          if (lane == 0) l_run = (hlf == 0 ? l_run * alpha : l_run) + ps;
        }
      }
      float mx = fmaxf(fabsf(wv[0]), fabsf(wv[1]));
      float os = ov[0] + ov[1];
      for (int off = 16; off > 0; off >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        os += __shfl_xor_sync(0xffffffffu, os, off);
      }
      const float inv = mx > 0.f ? kFix / mx : 0.f;
      // both tokens' 16-bit fixed-point values in one word: token lane | token lane+32 << 16
      const uint32_t pv = ((uint32_t)to_fix(wv[0], inv) & 0xFFFFu) | ((uint32_t)to_fix(wv[1], inv) << 16);
      uint32_t word = 0;
      if (r == 0) {
        // lane = word w (8) x kind k: tokens 8w + 2i + (k >> 1), byte hi (k even) or lo
        const int w8 = lane >> 2, k = lane & 3, half = w8 >> 2;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tk = 8 * w8 + 2 * i + (k >> 1);
          const uint32_t x = __shfl_sync(0xffffffffu, pv, tk & 31);
          const int v = (int)(int16_t)(x >> (16 * half));
          word |= ((k & 1) ? fix_lo(v) : fix_hi(v)) << (8 * i);
        }
      } else {
        // lane = word j (4) x mask m (4) x part: tokens 16j + 4i + m
        const int j = lane >> 3, m = (lane >> 1) & 3, part = lane & 1, half = j >> 1;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tk = 16 * j + 4 * i + m;
          const uint32_t x = __shfl_sync(0xffffffffu, pv, tk & 31);
          const int v = (int)(int16_t)(x >> (16 * half));
          word |= (part ? fix_lo(v) : fix_hi(v)) << (8 * i);
        }
      }
      pack_s[buf][item][lane] = word;
      if (lane == 0) {
        tau_s[buf][item] = mx / kFix;
        off_s[buf][item] = os;
      }
    }
    __syncthreads();                                   // B2: weight operands are in pack_s

    // ---- phase 2: value accumulation, thread = (channel, anchor | residual) ----
    if (p2_active) {
      const int gi = p2_ch / GS;
      float add = 0.f;
      if (p2_anchor) {
        const uint4* row = reinterpret_cast<const uint4*>(AV + p2_ch * (kTile / 2));
        const uint32_t* pw = pack_s[buf][gi];
        int eh = 0, el = 0, oh = 0, ol = 0;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint4 x4 = row[h2];
          const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int w = h2 * 4 + q4;
            const uint4 pk = *reinterpret_cast<const uint4*>(pw + 4 * w);
            const uint32_t lo4 = xs[q4] & 0x0F0F0F0Fu, hi4 = xs[q4] & 0xF0F0F0F0u;
            eh = dp4a_us(lo4, pk.x, eh);
            el = dp4a_uu(lo4, pk.y, el);
            oh = dp4a_us(hi4, pk.z, oh);
            ol = dp4a_uu(hi4, pk.w, ol);
          }
        }
        const int t = shl(shl(eh, 8) + el, 4) + shl(oh, 8) + ol;        // 16 x sum(w_fix * code)
        add = fmaf((float)t, tau_s[buf][gi] * (1.f / 16.f), off_s[buf][gi]);
      } else {
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const int item = (1 + r) * NG + gi;
          const uint32_t* pw = pack_s[buf][item];
          const uint4 x4 = *reinterpret_cast<const uint4*>(RES + (2 * r + 1) * C::R_TILE + p2_ch * (kTile / 4));
          const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w};
          int hm[4] = {0, 0, 0, 0}, lm[4] = {0, 0, 0, 0};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 pa = *reinterpret_cast<const uint4*>(pw + 8 * j);
            const uint4 pb = *reinterpret_cast<const uint4*>(pw + 8 * j + 4);
            const uint32_t b0 = xs[j] & 0x03030303u, b1 = xs[j] & 0x0C0C0C0Cu;
            const uint32_t b2 = xs[j] & 0x30303030u, b3 = xs[j] & 0xC0C0C0C0u;
            hm[0] = dp4a_us(b0, pa.x, hm[0]); lm[0] = dp4a_uu(b0, pa.y, lm[0]);
            hm[1] = dp4a_us(b1, pa.z, hm[1]); lm[1] = dp4a_uu(b1, pa.w, lm[1]);
            hm[2] = dp4a_us(b2, pb.x, hm[2]); lm[2] = dp4a_uu(b2, pb.y, lm[2]);
            hm[3] = dp4a_us(b3, pb.z, hm[3]); lm[3] = dp4a_uu(b3, pb.w, lm[3]);
          }
          const int t = shl(shl(hm[0], 8) + lm[0], 6) + shl(shl(hm[1], 8) + lm[1], 4) +
                        shl(shl(hm[2], 8) + lm[2], 2) + (shl(hm[3], 8) + lm[3]);   // 64 x sum
          add += fmaf((float)t, tau_s[buf][item] * (1.f / 64.f), off_s[buf][item]);
        }
      }
      acc = fmaf(acc, alpha, add);
    }
    // no barrier here: the next tile's writes go to the other parity buffers, and its
    // stage is refilled only after the next B1
  }

  if (aborted) {
    // let the copies still in flight land before the CTA exits (each wait bounded)
    if (tid == 0)
      for (long long v = fail_u; v < u1 && v < fail_u + STAGES; ++v)
        (void)mbar_wait_bounded(&full_bar[(v - u0) % STAGES], (uint32_t)(((v - u0) / STAGES) & 1));
    __syncthreads();
    return;
  }
  __syncthreads();
  if (cur_bh >= 0) flush(cur_bh);
}

template <int D, int GS, int NRES>
cudaError_t launch_t(const DecodeArgs& a, int grid, cudaStream_t stream) {
  using C = Cfg<D, GS, NRES>;
  auto k = decode_kernel<D, GS, NRES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k<<<grid, kThreads, C::SMEM, stream>>>(a);
  return cudaGetLastError();
}

template <int D, int GS>
cudaError_t launch_d(const DecodeArgs& a, int grid, int nres, cudaStream_t stream) {
  switch (nres) {
    case 0: return launch_t<D, GS, 0>(a, grid, stream);
    case 1: return launch_t<D, GS, 1>(a, grid, stream);
    case 2: return launch_t<D, GS, 2>(a, grid, stream);
    case 3: return launch_t<D, GS, 3>(a, grid, stream);
  }
  return cudaErrorNotSupported;
}

int pstride_for(int d) { return ((2 + 2 * d) + 3) / 4 * 4; }

}  // namespace

int decode_max_chained_loops() { return kMaxRes + 1; }

size_t decode_workspace_bytes(const Geom& g, int batch, int num_sms) {
  size_t C = (size_t)num_sms * kCtasPerSm;
  size_t bh = (size_t)batch * g.H;
  size_t counters = (bh * 4 + 255) / 256 * 256;
  return 256 + counters + (C + bh) * pstride_for(g.d) * sizeof(float);
}

cudaError_t launch_decode(const rq_cache& c, int layer, int group, int loop, int batch,
                          const __nv_bfloat16* q, const __nv_bfloat16* k_cur,
                          const __nv_bfloat16* v_cur, const int32_t* seq_lens, float scale,
                          float* out, void* workspace, cudaStream_t stream) {
  if (batch > kMaxRows) return cudaErrorInvalidValue;
  const int P = c.geom.P;
  const bool chained = c.geom.mode == RQ_MODE_CHAINED;
  const int nres = loop == P - 1 ? 0 : (chained ? P - 1 - loop : 1);
  if (nres > kMaxRes) return cudaErrorNotSupported;
  DecodeArgs a;
  a.g = c.geom;
  a.base = c.base;
  a.R = c.R;
  a.q = q;
  a.k_cur = k_cur;
  a.v_cur = v_cur;
  a.seq_lens = seq_lens;
  a.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<int32_t*>(ws);
  a.counters = reinterpret_cast<int32_t*>(ws + 256);
  size_t bh = (size_t)batch * c.geom.H;
  a.partials = reinterpret_cast<float*>(ws + 256 + (bh * 4 + 255) / 256 * 256);
  a.pstride = pstride_for(c.geom.d);
  a.layer = layer;
  a.group = group;
  a.batch = batch;
  a.res0 = loop;
  a.qscale = scale * kLog2e;
  const int grid = c.num_sms * kCtasPerSm;
  const int d = c.geom.d, gs = c.geom.g;
  if (d == 128 && gs == 32) return launch_d<128, 32>(a, grid, nres, stream);
  if (d == 128 && gs == 16) return launch_d<128, 16>(a, grid, nres, stream);
  if (d == 96 && gs == 32) return launch_d<96, 32>(a, grid, nres, stream);
  if (d == 96 && gs == 16) return launch_d<96, 16>(a, grid, nres, stream);
  return cudaErrorNotSupported;
}

}  // namespace rq

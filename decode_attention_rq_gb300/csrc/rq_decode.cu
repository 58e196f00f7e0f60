// rq_decode_attention: split-K decode attention over the compressed cache.
//
// The explainer "ResidualQuant stores looped-Transformer KV caches as 2-bit
// residuals" (paragraph on the custom attention kernel and the one on shared
// versus chained anchors) fixes what the kernel must do: rebuild each loop's
// K/V as c * anchor + residual tile by tile in on-chip memory, never writing
// the rebuilt tensor back, reading two planes per key for a non-anchor loop.
//
// GB300 design
//   * Work units are (row, head, 64-token tile).  A fixed grid of
//     num_SMs x kCtasPerSm CTAs takes equal contiguous ranges of the flattened
//     unit list (a range may cross (row, head) boundaries), so every SM
//     streams the same number of tiles whatever the batch and lengths.
//   * Each tile's four plane slices (anchor K/V, residual K/V of this loop)
//     are contiguous and 16-byte aligned; one thread issues 1-D TMA bulk
//     copies into a kStages-deep shared-memory ring, completion tracked by
//     mbarriers (bounded waits).
//   * Scores use the rotated query: q.(c a_hat + R^T r_hat) = c (q.a_hat) +
//     (R q).r_hat, so R is applied once per (row, head) segment to q, and the
//     value side accumulates the anchor part and the rotated residual part
//     separately; R^T is applied once, at the merge.
//   * Per-group algebra: q.x_hat over a group = s * sum(q * code) + o * sum(q).
//     V side: sum_j p_j c_j (s_jg code_jk + o_jg) keeps the offsets as one
//     scalar per (tile, group).
//   * Online softmax in base 2 (the scale * log2(e) is folded into q); each
//     CTA writes one partial (m, l, acc_anchor, acc_residual) per segment; the
//     last CTA to finish a (row, head) -- found with an atomic counter, no
//     spinning -- merges the partials, adds the current token from the BF16
//     temporary buffer, applies R^T and writes the output.
#include <cuda_fp8.h>

#include "rq_internal.cuh"

namespace rq {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 2;
constexpr int kStages = 4;
constexpr int kMaxRows = 256;          // batch rows one call may cover
constexpr float kLog2e = 1.4426950408889634f;

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
  int layer, group, loop, batch;
  float qscale;          // softmax_scale * log2(e)
};

template <int D>
struct PartialLayout {
  // m, l, then acc_a[D], acc_r[D]
  static constexpr int kStride = ((2 + 2 * D) + 3) / 4 * 4;
};

__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(__half(hr));
}

// flattened unit u -> CTA that owns it, for ranges [floor(cU/C), floor((c+1)U/C))
__device__ __forceinline__ int cta_of(long long u, long long U, int C) {
  return (int)(((u + 1) * C - 1) / U);
}
// CTA c's range [floor(cU/C), floor((c+1)U/C)) intersects [s0, s1) (ranges may be
// empty when there are fewer units than CTAs; such CTAs contribute nothing)
__device__ __forceinline__ bool contributes(int c, long long s0, long long s1, long long U, int C) {
  long long r0 = (long long)c * U / C, r1 = (long long)(c + 1) * U / C;
  return (r0 > s0 ? r0 : s0) < (r1 < s1 ? r1 : s1);
}

template <int D, int GS, bool HAS_RES>
struct Cfg {
  static constexpr int NG = D / GS;
  static constexpr int A_CODES = kTile * D / 2;
  static constexpr int R_CODES = kTile * D / 4;
  static constexpr int META = kTile * NG * 2;
  static constexpr int A_TILE = A_CODES + META;
  static constexpr int R_TILE = R_CODES + META + kTile * 2;
  static constexpr int STAGE = 2 * A_TILE + (HAS_RES ? 2 * R_TILE : 0);
  static constexpr int NPAIR = kTile * NG;                 // (token, group) pairs per tile
  static constexpr int PPT = (NPAIR + kThreads - 1) / kThreads;
  static constexpr int SMEM = kStages * STAGE;
};

template <int D, int GS, bool HAS_RES>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(DecodeArgs a) {
  using C = Cfg<D, GS, HAS_RES>;
  constexpr int NG = C::NG;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[kStages];
  __shared__ int pre_s[kMaxRows + 1];
  __shared__ int nt_s[kMaxRows];
  __shared__ float q_s[D], qr_s[D];
  __shared__ float part_s[NG][kTile];
  __shared__ float wa_s[NG][kTile], wr_s[NG][kTile], oa_s[NG][kTile], or_s[NG][kTile];
  __shared__ float offa_s[NG], offr_s[NG];
  __shared__ float red_s[8];
  __shared__ float m_sh, alpha_sh;
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

  // unit -> (bh, tile)
  auto locate = [&](long long u, int* bh, int* tile) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {   // last row b with pre_s[b] <= u
      int mid = (lo + hi + 1) >> 1;
      if (pre_s[mid] <= u) lo = mid; else hi = mid - 1;
    }
    int b = lo;
    int rem = (int)(u - pre_s[b]);
    *bh = b * H + rem / nt_s[b];
    *tile = rem % nt_s[b];
  };

  const int jres = a.loop;   // residual plane of this loop (shared mode)
  auto issue = [&](long long u, int stage) {
    int bh, tile;
    locate(u, &bh, &tile);
    const uint8_t* region = a.base + a.g.region_offset(a.layer, a.group, bh / H, bh % H);
    uint8_t* dst = smem + stage * C::STAGE;
    mbar_arrive_expect_tx(&full_bar[stage], C::STAGE);
    bulk_g2s(dst, region + a.g.anchor_plane(0) + (int64_t)tile * C::A_TILE, C::A_TILE, &full_bar[stage]);
    bulk_g2s(dst + C::A_TILE, region + a.g.anchor_plane(1) + (int64_t)tile * C::A_TILE, C::A_TILE,
             &full_bar[stage]);
    if (HAS_RES) {
      bulk_g2s(dst + 2 * C::A_TILE, region + a.g.res_plane(jres, 0) + (int64_t)tile * C::R_TILE,
               C::R_TILE, &full_bar[stage]);
      bulk_g2s(dst + 2 * C::A_TILE + C::R_TILE,
               region + a.g.res_plane(jres, 1) + (int64_t)tile * C::R_TILE, C::R_TILE,
               &full_bar[stage]);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full_bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < kStages && u0 + s < u1; ++s) issue(u0 + s, s);

  // per-thread state
  float qreg[C::PPT][GS], qrreg[C::PPT][GS], qsum[C::PPT], qrsum[C::PPT];
  float acc = 0.f;          // phase-2 accumulator: (channel, kind)
  float m_run = -INFINITY, l_run = 0.f;
  int cur_bh = -1;
  bool aborted = false;
  long long fail_u = 0;

  const int p2_ch = tid < D ? tid : tid - D;
  const bool p2_anchor = tid < D;
  const bool p2_active = tid < (HAS_RES ? 2 * D : D);

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
    // current token score, base-2 logits
    float sc = 0.f;
    for (int k = tid; k < D; k += kThreads)
      sc += q_s[k] * __bfloat162float(a.k_cur[(size_t)bh * D + k]);
    for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
    if (lane == 0) red_s[warp] = sc;
    __syncthreads();
    if (tid == 0) {
      float s_cur = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) s_cur += red_s[w];
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
      alpha_sh = L;
      red_s[0] = s_cur;
    }
    __syncthreads();
    const float M = m_sh, L = alpha_sh, s_cur = red_s[0];
    // accumulate partials: anchor part straight, residual part into qr_s (reused as scratch)
    if (tid < D) {
      float va = 0.f, vr = 0.f;
      for (int c = c_lo; c <= c_hi; ++c) {
        if (!contributes(c, s0, s1, U, Cn)) continue;
        const float* pc = a.partials + (size_t)(c + bh) * a.pstride;
        float w = exp2f(__ldcg(pc) - M);
        va = fmaf(w, __ldcg(pc + 2 + tid), va);
        if (HAS_RES) vr = fmaf(w, __ldcg(pc + 2 + D + tid), vr);
      }
      va = fmaf(exp2f(s_cur - M), __bfloat162float(a.v_cur[(size_t)bh * D + tid]), va);
      if (HAS_RES) qr_s[tid] = vr;
      q_s[tid] = va;   // q_s no longer needed for this segment
    }
    __syncthreads();
    if (tid < D) {
      float o = q_s[tid];
      if (HAS_RES) {
        float t = 0.f;
        for (int k = 0; k < D; ++k) t = fmaf(__ldg(a.R + (size_t)k * D + tid), qr_s[k], t);  // (R^T acc_r)
        o += t;
      }
      a.out[(size_t)bh * D + tid] = o / L;
    }
    if (tid == 0) a.counters[bh] = 0;
    __syncthreads();
  };

  auto begin_segment = [&](int bh) {
    // scaled query, rotated query, per-thread group registers
    for (int k = tid; k < D; k += kThreads) q_s[k] = __bfloat162float(a.q[(size_t)bh * D + k]) * a.qscale;
    __syncthreads();
    if (HAS_RES) {
      for (int i = tid; i < D; i += kThreads) {
        const float* Rrow = a.R + (size_t)i * D;
        float t = 0.f;
        for (int k = 0; k < D; ++k) t = fmaf(__ldg(Rrow + k), q_s[k], t);
        qr_s[i] = t;
      }
      __syncthreads();
    }
#pragma unroll
    for (int pp = 0; pp < C::PPT; ++pp) {
      int p = tid + pp * kThreads;
      int gi = p % NG;
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int k = 0; k < GS; ++k) {
        qreg[pp][k] = q_s[gi * GS + k];
        s1 += qreg[pp][k];
        qrreg[pp][k] = HAS_RES ? qr_s[gi * GS + k] : 0.f;
        s2 += qrreg[pp][k];
      }
      qsum[pp] = s1;
      qrsum[pp] = s2;
    }
    m_run = -INFINITY;
    l_run = 0.f;
    acc = 0.f;
    cur_bh = bh;
  };

  for (long long u = u0; u < u1; ++u) {
    const int it = (int)(u - u0), stage = it % kStages;
    int bh, tile;
    locate(u, &bh, &tile);
    if (bh != cur_bh) {
      if (cur_bh >= 0) flush(cur_bh);
      begin_segment(bh);
    }
    const int n_valid = min(kTile, a.seq_lens[bh / H] - tile * kTile);

    if (!mbar_wait_bounded(&full_bar[stage], (uint32_t)((it / kStages) & 1))) {
      if (tid == 0) atomicExch(&a.status[0], 1);
      aborted = true;
    }
    if (__syncthreads_or(aborted)) {
      aborted = true;
      fail_u = u;
      break;
    }

    const uint8_t* st = smem + stage * C::STAGE;
    const uint8_t* AK = st;
    const uint8_t* AV = st + C::A_TILE;
    const uint8_t* RK = st + 2 * C::A_TILE;
    const uint8_t* RV = RK + C::R_TILE;

    // ---- phase 1: partial score of each (token, group) pair ----
#pragma unroll
    for (int pp = 0; pp < C::PPT; ++pp) {
      int p = tid + pp * kThreads;
      if (p < C::NPAIR) {
        int gi = p % NG, tok = p / NG;
        // anchor codes of the group: GS nibbles
        const uint32_t* ak = reinterpret_cast<const uint32_t*>(AK + tok * (D / 2) + gi * (GS / 2));
        float dot = 0.f;
#pragma unroll
        for (int w = 0; w < GS / 8; ++w) {
          uint32_t x = ak[w];
#pragma unroll
          for (int n = 0; n < 8; ++n) dot = fmaf(qreg[pp][w * 8 + n], (float)((x >> (4 * n)) & 15u), dot);
        }
        uint16_t mk = *reinterpret_cast<const uint16_t*>(AK + C::A_CODES + tok * NG * 2 + gi * 2);
        float sa = e4m3_to_f32(mk & 0xFF), oa = e4m3_to_f32(mk >> 8);
        float score = fmaf(sa, dot, oa * qsum[pp]);
        if (HAS_RES) {
          const uint32_t* rk = reinterpret_cast<const uint32_t*>(RK + tok * (D / 4) + gi * (GS / 4));
          float dr = 0.f;
#pragma unroll
          for (int w = 0; w < GS / 16; ++w) {
            uint32_t x = rk[w];
#pragma unroll
            for (int n = 0; n < 16; ++n) dr = fmaf(qrreg[pp][w * 16 + n], (float)((x >> (2 * n)) & 3u), dr);
          }
          uint16_t mr = *reinterpret_cast<const uint16_t*>(RK + C::R_CODES + tok * NG * 2 + gi * 2);
          float sr = e4m3_to_f32(mr & 0xFF), orr = e4m3_to_f32(mr >> 8);
          uint16_t cb = *reinterpret_cast<const uint16_t*>(RK + C::R_CODES + C::META + tok * 2);
          score = fmaf(bf16_bits_to_f32(cb), score, fmaf(sr, dr, orr * qrsum[pp]));
        }
        part_s[gi][tok] = score;
      }
    }
    __syncthreads();

    // ---- softmax update over the tile (threads 0..63 own one token each) ----
    float s_tok = -INFINITY;
    if (tid < kTile) {
      if (tid < n_valid) {
        s_tok = 0.f;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) s_tok += part_s[gi][tid];
      }
      float mx = s_tok;
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0) red_s[warp] = mx;
    }
    __syncthreads();
    const float m_tile = fmaxf(red_s[0], red_s[1]);
    const float m_new = fmaxf(m_run, m_tile);
    const float alpha = exp2f(m_run - m_new);   // 0 on the first tile (m_run = -inf)
    float p_tok = 0.f;
    if (tid < kTile) {
      p_tok = tid < n_valid ? exp2f(s_tok - m_new) : 0.f;
      float ps = p_tok;
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      if (lane == 0) red_s[2 + warp] = ps;
      part_s[0][tid] = p_tok;   // reuse: p per token
    }
    __syncthreads();
    l_run = l_run * alpha + red_s[2] + red_s[3];
    m_run = m_new;

    // ---- value weights per (token, group) and offset sums per group ----
#pragma unroll
    for (int pp = 0; pp < C::PPT; ++pp) {
      int p = tid + pp * kThreads;
      if (p < C::NPAIR) {
        int gi = p % NG, tok = p / NG;
        float pt = part_s[0][tok];
        float wa = 0.f, oa = 0.f, wr = 0.f, orr = 0.f;
        if (tok < n_valid) {
          uint16_t mv = *reinterpret_cast<const uint16_t*>(AV + C::A_CODES + tok * NG * 2 + gi * 2);
          float cv = 1.f;
          if (HAS_RES) {
            uint16_t cb = *reinterpret_cast<const uint16_t*>(RV + C::R_CODES + C::META + tok * 2);
            cv = bf16_bits_to_f32(cb);
            uint16_t mr = *reinterpret_cast<const uint16_t*>(RV + C::R_CODES + tok * NG * 2 + gi * 2);
            wr = pt * e4m3_to_f32(mr & 0xFF);
            orr = pt * e4m3_to_f32(mr >> 8);
          }
          wa = pt * cv * e4m3_to_f32(mv & 0xFF);
          oa = pt * cv * e4m3_to_f32(mv >> 8);
        }
        wa_s[gi][tok] = wa;
        wr_s[gi][tok] = wr;
        oa_s[gi][tok] = oa;
        or_s[gi][tok] = orr;
      }
    }
    __syncthreads();
    if (warp < NG) {   // warp gi sums the group's offset terms over the 64 tokens
      float x = oa_s[warp][lane] + oa_s[warp][lane + 32];
      float y = or_s[warp][lane] + or_s[warp][lane + 32];
      for (int off = 16; off > 0; off >>= 1) {
        x += __shfl_xor_sync(0xffffffffu, x, off);
        y += __shfl_xor_sync(0xffffffffu, y, off);
      }
      if (lane == 0) { offa_s[warp] = x; offr_s[warp] = y; }
    }
    __syncthreads();

    // ---- phase 2: value accumulation, thread = (channel, anchor|residual) ----
    if (p2_active) {
      const int gi = p2_ch / GS;
      acc *= alpha;
      if (p2_anchor) {
        const uint32_t* row = reinterpret_cast<const uint32_t*>(AV + p2_ch * (kTile / 2));
#pragma unroll
        for (int w = 0; w < kTile / 8; ++w) {
          uint32_t x = row[w];
#pragma unroll
          for (int n = 0; n < 8; ++n) acc = fmaf(wa_s[gi][w * 8 + n], (float)((x >> (4 * n)) & 15u), acc);
        }
        acc += offa_s[gi];
      } else {
        const uint32_t* row = reinterpret_cast<const uint32_t*>(RV + p2_ch * (kTile / 4));
#pragma unroll
        for (int w = 0; w < kTile / 16; ++w) {
          uint32_t x = row[w];
#pragma unroll
          for (int n = 0; n < 16; ++n) acc = fmaf(wr_s[gi][w * 16 + n], (float)((x >> (2 * n)) & 3u), acc);
        }
        acc += offr_s[gi];
      }
    }
    __syncthreads();   // stage fully consumed
    if (tid == 0 && u + kStages < u1) issue(u + kStages, stage);
  }

  if (aborted) {
    // let the copies still in flight land before the CTA exits (each wait bounded)
    if (tid == 0)
      for (long long v = fail_u; v < u1 && v < fail_u + kStages; ++v)
        (void)mbar_wait_bounded(&full_bar[(v - u0) % kStages], (uint32_t)(((v - u0) / kStages) & 1));
    __syncthreads();
    return;
  }
  if (cur_bh >= 0) flush(cur_bh);
}

template <int D, int GS, bool HAS_RES>
cudaError_t launch_t(const DecodeArgs& a, int grid, cudaStream_t stream) {
  using C = Cfg<D, GS, HAS_RES>;
  auto k = decode_kernel<D, GS, HAS_RES>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, C::SMEM, stream>>>(a);
  return cudaGetLastError();
}

template <int D, int GS>
cudaError_t launch_d(const DecodeArgs& a, int grid, bool has_res, cudaStream_t stream) {
  return has_res ? launch_t<D, GS, true>(a, grid, stream) : launch_t<D, GS, false>(a, grid, stream);
}

}  // namespace

static int pstride_for(int d) { return ((2 + 2 * d) + 3) / 4 * 4; }

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
  if (c.geom.mode != RQ_MODE_SHARED) return cudaErrorNotSupported;
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
  a.loop = loop;
  a.batch = batch;
  a.qscale = scale * kLog2e;
  const bool has_res = loop < c.geom.P - 1;
  const int grid = c.num_sms * kCtasPerSm;
  const int d = c.geom.d, gs = c.geom.g;
  if (d == 128 && gs == 32) return launch_d<128, 32>(a, grid, has_res, stream);
  if (d == 128 && gs == 16) return launch_d<128, 16>(a, grid, has_res, stream);
  if (d == 96 && gs == 32) return launch_d<96, 32>(a, grid, has_res, stream);
  if (d == 96 && gs == 16) return launch_d<96, 16>(a, grid, has_res, stream);
  return cudaErrorNotSupported;
}

}  // namespace rq

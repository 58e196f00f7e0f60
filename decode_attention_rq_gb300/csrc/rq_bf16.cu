// rq_decode_attention_bf16: the uncompressed comparator.
//
// The ai4snews summary of the ResidualQuant paper (throughput paragraph)
// measures against BF16 decode attention (vLLM FlashAttention); this library
// ships its own BF16 split-K decode kernel with the same structure as the
// compressed one -- balanced (row, head, 64-token tile) ranges per CTA, 1-D
// TMA bulk copies into a shared-memory ring, base-2 online softmax, last-CTA
// merge with the current token -- so the two differ only in what they read.
#include "rq_internal.cuh"

namespace rq {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 2;
constexpr int kStages = 3;
constexpr int kMaxRows = RQ_MAX_DECODE_BATCH;
constexpr float kLog2e = 1.4426950408889634f;

struct Bf16Args {
  const __nv_bfloat16 *k, *v, *k_cur, *v_cur, *q;
  const int32_t* seq_lens;
  float* out;
  int32_t* status;
  int32_t* counters;
  float* partials;
  int pstride, batch, H, max_seq;
  float qscale;
};

// Balanced split of U units over C CTAs: CTA c takes [start(c), start(c+1)) with
// start(c) = c*q + min(c, rem), q = U / C, rem = U % C (32-bit arithmetic only).
struct Split {
  int q, rem;
  __device__ __forceinline__ int start(int c) const { return c * q + min(c, rem); }
  __device__ __forceinline__ int owner(int u) const {
    const int big = (q + 1) * rem;
    return u < big ? u / (q + 1) : rem + (u - big) / q;
  }
};

__device__ __forceinline__ float2 bf2_to_f2(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

template <int D>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) bf16_kernel(Bf16Args a) {
  constexpr int ROW = D * 2;                  // bytes per token row
  constexpr int TILE = kTile * ROW;           // bytes per K (or V) tile
  constexpr int STAGE = 2 * TILE;
  constexpr int NC = D / 32;                  // 16-byte chunks per quarter row
  constexpr int NPAIR2 = (D / 2) * 4;         // (channel pair, token quarter) threads
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[kStages];
  __shared__ int pre_s[kMaxRows + 1], nt_s[kMaxRows];
  __shared__ __align__(16) float q_s[D];
  __shared__ float part_s[4][kTile];
  __shared__ float p_s[kTile];
  __shared__ float acc_s[4][D];
  __shared__ float red_s[8];
  __shared__ float m_sh, l_sh;
  __shared__ int flag_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, B = a.batch;
  const int Cn = gridDim.x, cta = blockIdx.x;

  for (int b = tid; b < B; b += kThreads) {
    int n = a.seq_lens[b];
    n = n < 0 ? 0 : (n > a.max_seq ? a.max_seq : n);
    nt_s[b] = (n + kTile - 1) / kTile;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) { pre_s[b] = acc; acc += H * nt_s[b]; }
    pre_s[B] = acc;
  }
  __syncthreads();
  const int U = pre_s[B];
  for (int bh = cta; bh < B * H; bh += Cn) {
    if (nt_s[bh / H] != 0) continue;
    for (int k = tid; k < D; k += kThreads)
      a.out[(size_t)bh * D + k] = __bfloat162float(a.v_cur[(size_t)bh * D + k]);
  }
  if (U == 0) return;
  const Split split{U / Cn, U % Cn};
  const int u0 = split.start(cta), u1 = split.start(cta + 1);
  if (u0 >= u1) return;

  auto locate = [&](int u, int* bh, int* tile) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (pre_s[mid] <= u) lo = mid; else hi = mid - 1;
    }
    int rem = (int)(u - pre_s[lo]);
    *bh = lo * H + rem / nt_s[lo];
    *tile = rem % nt_s[lo];
  };
  auto rows_of = [&](int bh, int tile) {
    return min(kTile, min(a.max_seq, a.seq_lens[bh / H]) - tile * kTile);
  };
  auto issue = [&](int u, int stage) {
    int bh, tile;
    locate(u, &bh, &tile);
    // copy only the rows that exist in the caller's buffer (and are valid)
    uint32_t bytes = (uint32_t)rows_of(bh, tile) * ROW;
    size_t off = ((size_t)bh * a.max_seq + (size_t)tile * kTile) * D;
    uint8_t* dst = smem + stage * STAGE;
    mbar_arrive_expect_tx(&full_bar[stage], 2 * bytes);
    bulk_g2s(dst, a.k + off, bytes, &full_bar[stage]);
    bulk_g2s(dst + TILE, a.v + off, bytes, &full_bar[stage]);
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full_bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < kStages && u0 + s < u1; ++s) issue(u0 + s, s);

  float m_run = -INFINITY, l_run = 0.f;
  float acc0 = 0.f, acc1 = 0.f;
  int cur_bh = -1;
  bool aborted = false;
  int fail_u = 0;
  const int tok1 = tid % kTile, part1 = tid / kTile;      // phase 1: (token, quarter row)
  const int ch2 = tid % (D / 2), qt2 = tid / (D / 2);     // phase 2: (channel pair, token quarter)
  const bool p2_active = tid < NPAIR2;

  auto flush = [&](int bh) {
    if (p2_active) { acc_s[qt2][2 * ch2] = acc0; acc_s[qt2][2 * ch2 + 1] = acc1; }
    __syncthreads();
    float* part = a.partials + (size_t)(cta + bh) * a.pstride;
    if (tid == 0) { part[0] = m_run; part[1] = l_run; }
    if (tid < D) part[2 + tid] = acc_s[0][tid] + acc_s[1][tid] + acc_s[2][tid] + acc_s[3][tid];
    __threadfence();
    __syncthreads();
    const int b = bh / H, h = bh % H;
    const int s0 = pre_s[b] + h * nt_s[b], s1 = s0 + nt_s[b];
    const int c_lo = split.owner(s0), c_hi = split.owner(s1 - 1);
    if (tid == 0) flag_s = (atomicAdd(&a.counters[bh], 1) == c_hi - c_lo);
    __syncthreads();
    if (!flag_s) return;
    __threadfence();
    float sc = 0.f;
    for (int k = tid; k < D; k += kThreads) sc += q_s[k] * __bfloat162float(a.k_cur[(size_t)bh * D + k]);
    for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
    if (lane == 0) red_s[warp] = sc;
    __syncthreads();
    if (tid == 0) {
      float s_cur = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) s_cur += red_s[w];
      float M = s_cur;
      for (int c = c_lo; c <= c_hi; ++c) M = fmaxf(M, __ldcg(a.partials + (size_t)(c + bh) * a.pstride));
      float L = exp2f(s_cur - M);
      for (int c = c_lo; c <= c_hi; ++c) {
        const float* pc = a.partials + (size_t)(c + bh) * a.pstride;
        L += __ldcg(pc + 1) * exp2f(__ldcg(pc) - M);
      }
      m_sh = M; l_sh = L; red_s[0] = s_cur;
    }
    __syncthreads();
    if (tid < D) {
      const float M = m_sh;
      float o = exp2f(red_s[0] - M) * __bfloat162float(a.v_cur[(size_t)bh * D + tid]);
      for (int c = c_lo; c <= c_hi; ++c) {
        const float* pc = a.partials + (size_t)(c + bh) * a.pstride;
        o = fmaf(exp2f(__ldcg(pc) - M), __ldcg(pc + 2 + tid), o);
      }
      a.out[(size_t)bh * D + tid] = o / l_sh;
    }
    if (tid == 0) a.counters[bh] = 0;
    __syncthreads();
  };

  for (int u = u0; u < u1; ++u) {
    const int it = (int)(u - u0), stage = it % kStages;
    int bh, tile;
    locate(u, &bh, &tile);
    if (bh != cur_bh) {
      if (cur_bh >= 0) flush(cur_bh);
      for (int k = tid; k < D; k += kThreads) q_s[k] = __bfloat162float(a.q[(size_t)bh * D + k]) * a.qscale;
      m_run = -INFINITY; l_run = 0.f; acc0 = acc1 = 0.f;
      cur_bh = bh;
      __syncthreads();
    }
    const int n_valid = rows_of(bh, tile);
    if (!mbar_wait_bounded(&full_bar[stage], (uint32_t)((it / kStages) & 1))) {
      if (tid == 0) atomicExch(&a.status[0], 1);
      aborted = true;
    }
    if (__syncthreads_or(aborted)) { aborted = true; fail_u = u; break; }
    const uint8_t* Ks = smem + stage * STAGE;
    const uint8_t* Vs = Ks + TILE;

    // phase 1: quarter-row dot products; chunk order rotated by token to spread banks
    {
      float dot = 0.f;
      if (tok1 < n_valid) {
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          int chunk = part1 * NC + (i + tok1) % NC;
          uint4 kk = *reinterpret_cast<const uint4*>(Ks + tok1 * ROW + chunk * 16);
          float4 qa = *reinterpret_cast<const float4*>(q_s + chunk * 8);
          float4 qb = *reinterpret_cast<const float4*>(q_s + chunk * 8 + 4);
          float2 k0 = bf2_to_f2(kk.x), k1 = bf2_to_f2(kk.y), k2 = bf2_to_f2(kk.z), k3 = bf2_to_f2(kk.w);
          dot = fmaf(qa.x, k0.x, dot); dot = fmaf(qa.y, k0.y, dot);
          dot = fmaf(qa.z, k1.x, dot); dot = fmaf(qa.w, k1.y, dot);
          dot = fmaf(qb.x, k2.x, dot); dot = fmaf(qb.y, k2.y, dot);
          dot = fmaf(qb.z, k3.x, dot); dot = fmaf(qb.w, k3.y, dot);
        }
      }
      part_s[part1][tok1] = dot;
    }
    __syncthreads();
    float s_tok = -INFINITY;
    if (tid < kTile) {
      if (tid < n_valid) s_tok = part_s[0][tid] + part_s[1][tid] + part_s[2][tid] + part_s[3][tid];
      float mx = s_tok;
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0) red_s[warp] = mx;
    }
    __syncthreads();
    const float m_new = fmaxf(m_run, fmaxf(red_s[0], red_s[1]));
    const float alpha = ex2_fast(m_run - m_new);
    if (tid < kTile) {
      float p = tid < n_valid ? ex2_fast(s_tok - m_new) : 0.f;
      p_s[tid] = p;
      for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
      if (lane == 0) red_s[2 + warp] = p;
    }
    __syncthreads();
    l_run = l_run * alpha + red_s[2] + red_s[3];
    m_run = m_new;

    // phase 2: thread = (channel pair, quarter of the tile's tokens)
    if (p2_active) {
      acc0 *= alpha;
      acc1 *= alpha;
      const int t0 = qt2 * (kTile / 4);
      const int t1 = min(t0 + kTile / 4, n_valid);
      for (int t = t0; t < t1; ++t) {
        float2 v = bf2_to_f2(*reinterpret_cast<const uint32_t*>(Vs + t * ROW + ch2 * 4));
        float p = p_s[t];
        acc0 = fmaf(p, v.x, acc0);
        acc1 = fmaf(p, v.y, acc1);
      }
    }
    __syncthreads();
    if (tid == 0 && u + kStages < u1) issue(u + kStages, stage);
  }
  if (aborted) {
    if (tid == 0)
      for (int v = fail_u; v < u1 && v < fail_u + kStages; ++v)
        (void)mbar_wait_bounded(&full_bar[(v - u0) % kStages], (uint32_t)(((v - u0) / kStages) & 1));
    __syncthreads();
    return;
  }
  if (cur_bh >= 0) flush(cur_bh);
}

template <int D>
cudaError_t launch_t(const Bf16Args& a, int grid, cudaStream_t stream) {
  constexpr int SMEM = kStages * 2 * kTile * D * 2;
  cudaError_t e = cudaFuncSetAttribute(bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  bf16_kernel<D><<<grid, kThreads, SMEM, stream>>>(a);
  return cudaGetLastError();
}

int pstride_for(int d) { return ((2 + d) + 3) / 4 * 4; }

}  // namespace

size_t bf16_workspace_bytes(int batch, int heads, int d, int num_sms) {
  size_t C = (size_t)num_sms * kCtasPerSm, bh = (size_t)batch * heads;
  return 256 + (bh * 4 + 255) / 256 * 256 + (C + bh) * pstride_for(d) * sizeof(float);
}

cudaError_t launch_bf16(const __nv_bfloat16* k, const __nv_bfloat16* v, const __nv_bfloat16* k_cur,
                        const __nv_bfloat16* v_cur, const __nv_bfloat16* q, const int32_t* seq_lens,
                        int batch, int heads, int d, int max_seq, float scale, float* out,
                        void* workspace, int num_sms, cudaStream_t stream) {
  if (batch > kMaxRows) return cudaErrorInvalidValue;
  Bf16Args a;
  a.k = k; a.v = v; a.k_cur = k_cur; a.v_cur = v_cur; a.q = q;
  a.seq_lens = seq_lens;
  a.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  size_t bh = (size_t)batch * heads;
  a.status = reinterpret_cast<int32_t*>(ws);
  a.counters = reinterpret_cast<int32_t*>(ws + 256);
  a.partials = reinterpret_cast<float*>(ws + 256 + (bh * 4 + 255) / 256 * 256);
  a.pstride = pstride_for(d);
  a.batch = batch; a.H = heads; a.max_seq = max_seq;
  a.qscale = scale * kLog2e;
  const int grid = num_sms * kCtasPerSm;
  if (d == 128) return launch_t<128>(a, grid, stream);
  if (d == 96) return launch_t<96>(a, grid, stream);
  return cudaErrorNotSupported;
}

}  // namespace rq

// rq_append: compress new tokens of one (layer, loop group) into the cache.
//
// Follows the stored-overlay paragraph of the explainer "ResidualQuant stores
// looped-Transformer KV caches as 2-bit residuals": the group's last loop is
// the INT4 anchor; every earlier loop l stores c_l (BF16 least-squares
// coefficient against the dequantized anchor, or in chained mode against the
// rebuilt loop l+1), and the 2-bit code of u_l = R (kv_l - c_l * ref).
// Group quantizer per rq.h: E4M3 offset = min, E4M3 scale = range / (2^b-1),
// code = exact nearest grid point, ties to even.
//
// Precision: every decision that fixes a stored byte (min/max, the E4M3
// roundings, the nearest code, the BF16 coefficient) is taken exactly, so
// stored bytes match the exact-arithmetic reading for a given rotated
// residual.  Each decision is first taken in float32 together with a bound
// on its rounding error; only when the bound does not rule out the other
// side of a rounding boundary is it retaken in float64 (FP64 throughput is a
// small fraction of FP32 on this GPU).  The rotation itself (d x d per
// vector) runs in float32 FMA.
//
// Grid: x = aligned block of 16 positions of one row, y = row * H + head,
// z = K/V (and, for short appends in shared mode, the residual loop: the
// loops are coded independently against the anchor, so each CTA takes one
// and requantizes the anchor as its reference; only loop 0's CTA writes the
// anchor plane).  A channel-major V word holds 8 (INT4) or 16 (INT2)
// aligned positions, so the words a CTA rewrites are touched by no other CTA
// that writes the same plane.
#include "rq_quant.cuh"

namespace rq {
namespace {

constexpr int kThreads = 128;      // one thread per channel (d <= 128)
constexpr int kTok = 16;           // positions per CTA (an aligned block)

struct AppendArgs {
  Geom g;
  uint8_t* base;
  const float* R;
  const __nv_bfloat16* kv;
  const int32_t* seq_lens;
  int32_t* status;
  int layer, group, batch, n;
};

__device__ __forceinline__ float load_x(const AppendArgs& a, int p, int kvi, int b, int h, int t,
                                        int k) {
  size_t idx = ((((size_t)p * 2 + kvi) * a.batch + b) * a.g.H + h) * (size_t)a.n + t;
  return __bfloat162float(a.kv[idx * a.g.d + k]);
}

// Write the codes / metadata (and c) of the CTA's tokens into one plane; `tile`
// is that plane's tile holding positions p0 .. p0 + kTok - 1 (one tile: p0 is a
// multiple of kTok, which divides kTile).
__device__ void write_plane(const AppendArgs& a, uint8_t* tile, int64_t codes_bytes, int bits, bool channel_major,
                            int p0,
                            const bool* valid, const uint8_t (*codes)[128],
                            const uint16_t (*meta)[8], const uint16_t* cbits) {
  const int d = a.g.d, ng = a.g.ng, tid = threadIdx.x;
  const int per_byte = 8 / bits;
  if (!channel_major) {
    // token-major rows: thread handles byte `tid` of every token row
    const int row_bytes = d / per_byte;
    for (int t = 0; t < kTok; ++t) {
      if (!valid[t] || tid >= row_bytes) continue;
      int pos = p0 + t;
      uint8_t* row = tile + (pos % kTile) * row_bytes;
      uint32_t byte = 0;
      for (int m = 0; m < per_byte; ++m) byte |= (uint32_t)codes[t][tid * per_byte + m] << (bits * m);
      row[tid] = (uint8_t)byte;
    }
  } else {
    // channel-major rows: thread = channel; a 32-bit word holds tpw aligned positions,
    // position q of the word in byte q % 4 at bit field q / 4
    if (tid < d) {
      const int row_bytes = kTile / per_byte;
      const int tpw = 4 * per_byte;
      const uint32_t fmask = (1u << bits) - 1u;
      for (int t0 = 0; t0 < kTok; t0 += tpw) {
        bool any = false;
        for (int q = 0; q < tpw; ++q) any |= valid[t0 + q];
        if (!any) continue;
        const int pos0 = p0 + t0;   // word-aligned: p0 is a multiple of kTok
        uint32_t* wp = reinterpret_cast<uint32_t*>(tile + tid * row_bytes + (pos0 % kTile) / per_byte);
        uint32_t word = *wp;
        for (int q = 0; q < tpw; ++q) {
          if (!valid[t0 + q]) continue;
          const int sh = 8 * (q & 3) + bits * (q >> 2);
          word = (word & ~(fmask << sh)) | ((uint32_t)codes[t0 + q][tid] << sh);
        }
        *wp = word;
      }
    }
  }
  // metadata (scale, offset) per group, and c
  for (int i = tid; i < kTok * ng; i += kThreads) {
    int t = i / ng, gi = i % ng;
    if (!valid[t]) continue;
    int pos = p0 + t;
    *reinterpret_cast<uint16_t*>(tile + codes_bytes + (pos % kTile) * ng * 2 + gi * 2) = meta[t][gi];
  }
  if (cbits) {
    for (int t = tid; t < kTok; t += kThreads) {
      if (!valid[t]) continue;
      int pos = p0 + t;
      *reinterpret_cast<uint16_t*>(tile + codes_bytes + a.g.meta + (pos % kTile) * 2) = cbits[t];
    }
  }
}

// u[t][i] = sum_k R[i][k] e[t][k] for the first NT token slots; thread = output
// channel i; the sum runs k = 0..D-1 as a chain of float32 fused multiply-adds.
// The row of R is loaded first, all of it in flight.
template <int NT, int D>
__device__ __forceinline__ void rotate_rows(const float* R, int i, const float (*e)[128],
                                            float (*u)[128]) {
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
  const float4* Rrow = reinterpret_cast<const float4*>(R + (size_t)i * D);
  float4 rr[D / 4];
#pragma unroll
  for (int k4 = 0; k4 < D / 4; ++k4) rr[k4] = __ldg(Rrow + k4);
#pragma unroll
  for (int k4 = 0; k4 < D / 4; ++k4) {
    const float4 r = rr[k4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float4 x = *reinterpret_cast<const float4*>(&e[t][4 * k4]);
      acc[t] = fmaf(r.x, x.x, acc[t]);
      acc[t] = fmaf(r.y, x.y, acc[t]);
      acc[t] = fmaf(r.z, x.z, acc[t]);
      acc[t] = fmaf(r.w, x.w, acc[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) u[t][i] = acc[t];
}

// u[t] = H e[t] / sqrt(128) for the first NT token slots (RQ_MODE_HADAMARD, d =
// 128, thread = channel); every thread of the CTA calls it.  scratch: NT x 128
// floats of shared memory, may be u itself.
template <int NT>
__device__ __forceinline__ void hadamard_rows(int i, const float (*e)[128], float (*u)[128], float* scratch) {
  float v[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) v[t] = e[t][i];
  hadamard128<NT>(v, i, scratch);
#pragma unroll
  for (int t = 0; t < NT; ++t) u[t][i] = v[t];
}

template <int D>
__global__ void __launch_bounds__(kThreads) append_kernel(AppendArgs a) {
  constexpr int d = D;
  const int gs = a.g.g, P = a.g.P, tid = threadIdx.x;
  const int b = blockIdx.y / a.g.H, h = blockIdx.y % a.g.H;
  const int kvi = blockIdx.z & 1, jz = blockIdx.z >> 1;
  const bool split = gridDim.z > 2;   // this CTA codes residual loop jz only
  const bool chained = (a.g.mode & RQ_MODE_CHAINED) != 0;
  const bool norm_ratio = (a.g.mode & RQ_MODE_NORM_RATIO) != 0;
  const bool hadamard = (a.g.mode & RQ_MODE_HADAMARD) != 0;   // d = 128: every thread is a channel

  __shared__ float ref_s[kTok][128];     // anchor_hat (shared) or rebuilt loop l+1 (chained)
  __shared__ float x_s[kTok][128];       // current loop, then its residual
  __shared__ float u_s[kTok][128];       // rotated residual
  __shared__ uint8_t codes_s[kTok][128];
  __shared__ uint16_t meta_s[kTok][8];
  __shared__ uint16_t c_s[kTok];
  __shared__ float cb_s[kTok];
  __shared__ bool valid_s[kTok];

  // launched as a programmatic dependent: seq_lens and kv may come from the kernel
  // ahead of this one.  It writes the cache, so it does not release the next
  // kernel early: that one starts once this kernel has finished.
  pdl_wait();
  const int start = a.seq_lens[b];
  if (start < 0 || start + a.n > a.g.Nmax) {
    if (blockIdx.x == 0 && h == 0 && blockIdx.z == 0 && tid == 0 && a.status) atomicExch(&a.status[1], 1);
    return;
  }
  const int blk = start / kTok + blockIdx.x;
  if (blk > (start + a.n - 1) / kTok) return;
  const int p0 = blk * kTok;
  if (tid < kTok) {
    int pos = p0 + tid;
    valid_s[tid] = pos >= start && pos < start + a.n;
  }
  for (int i = tid; i < kTok * 128; i += kThreads) {   // defined values in unused slots
    (&ref_s[0][0])[i] = 0.f;
    cb_s[i % kTok] = 0.f;
  }
  __syncthreads();

  // the tile of the CTA's block (paged layout: its page; a bad table entry skips the block)
  int page = 0;
  if (a.g.paged) {
    page = checked_page(a.g, raw_page(a.g, b, p0 / kTile), a.status);
    if (page < 0) return;   // every thread of the CTA reads the same entry
  }
  auto tile_ptr = [&](bool anchor, int j, int kv) {
    return a.base + a.g.tile_offset(a.layer, a.group, b, h, anchor, j, kv, p0 / kTile, page);
  };
  // all valid slots inside one aligned quad (a short append): rotate 4 slots, not 16
  int t_lo = kTok, t_hi = 0;
  for (int t = 0; t < kTok; ++t)
    if (valid_s[t]) { t_lo = min(t_lo, t); t_hi = t; }
  const int t4 = t_lo & ~3;   // t_lo < kTok: the block holds at least one appended position
  const bool few = t_hi < t4 + 4;
  const bool act = tid < d;
  if (split && act)   // this CTA's loop, loaded together with the anchor below
    for (int t = 0; t < kTok; ++t)
      x_s[t][tid] = valid_s[t] ? load_x(a, jz, kvi, b, h, p0 + t - start, tid) : 0.f;

  // ---- anchor: loop P-1, 4-bit (slots outside the appended range are skipped) ----
  for (int t = 0; t < kTok; ++t) {
    if (!valid_s[t]) continue;   // same for every thread of the CTA
    float v = act ? load_x(a, P - 1, kvi, b, h, p0 + t - start, tid) : 0.f;
    uint8_t sb, ob;
    float vh;
    int code = quantize_lane(v, act, gs, 15, &sb, &ob, &vh);
    if (act) {
      codes_s[t][tid] = (uint8_t)code;
      ref_s[t][tid] = vh;
      if (tid % gs == 0) meta_s[t][tid / gs] = (uint16_t)sb | ((uint16_t)ob << 8);
    }
  }
  __syncthreads();
  if (!split || jz == 0)
    write_plane(a, tile_ptr(true, 0, kvi), a.g.a_codes, 4, kvi == 1, p0, valid_s,
                codes_s, meta_s, nullptr);
  __syncthreads();

  // ---- earlier loops: shared mode any order; chained from P-2 down ----
  for (int j = P - 2; j >= 0; --j) {
    if (split && j != jz) continue;   // uniform over the CTA
    if (act && !split)
      for (int t = 0; t < kTok; ++t)
        x_s[t][tid] = valid_s[t] ? load_x(a, j, kvi, b, h, p0 + t - start, tid) : 0.f;
    __syncthreads();
    // coefficient per token (least squares or norm ratio), one warp per token
    {
      const int warp = tid / 32, lane = tid % 32;
      for (int t = warp; t < kTok; t += kThreads / 32) {
        if (!valid_s[t]) continue;   // same for every lane of the warp
        const uint16_t bits = coefficient_bits(x_s[t], ref_s[t], d, norm_ratio, lane);
        if (lane == 0) {
          c_s[t] = bits;
          cb_s[t] = bf16_bits_to_f32(bits);
        }
      }
    }
    __syncthreads();
    // residual e = x - cb * ref (float32, one rounding)
    if (act)
      for (int t = 0; t < kTok; ++t) x_s[t][tid] = fmaf(-cb_s[t], ref_s[t][tid], x_s[t][tid]);
    __syncthreads();
    // rotation u = R e, thread = output channel: a sequential FMA chain over k,
    // or the fast Walsh-Hadamard transform
    if (hadamard) {
      if (few) hadamard_rows<4>(tid, x_s + t4, u_s + t4, &u_s[t4][0]);
      else hadamard_rows<kTok>(tid, x_s, u_s, &u_s[0][0]);
    } else if (act) {
      if (few) rotate_rows<4, D>(a.R, tid, x_s + t4, u_s + t4);
      else rotate_rows<kTok, D>(a.R, tid, x_s, u_s);
    }
    __syncthreads();
    // 2-bit quantization of u
    for (int t = 0; t < kTok; ++t) {
      if (!valid_s[t]) continue;
      float v = act ? u_s[t][tid] : 0.f;
      uint8_t sb, ob;
      float vh;
      int code = quantize_lane(v, act, gs, 3, &sb, &ob, &vh);
      if (act) {
        codes_s[t][tid] = (uint8_t)code;
        u_s[t][tid] = vh;                     // r_hat, for the chained rebuild
        if (tid % gs == 0) meta_s[t][tid / gs] = (uint16_t)sb | ((uint16_t)ob << 8);
      }
    }
    __syncthreads();
    write_plane(a, tile_ptr(false, j, kvi), a.g.r_codes, 2, kvi == 1, p0,
                valid_s, codes_s, meta_s, c_s);
    if (chained && j > 0) {
      // rebuilt loop j = cb * ref + R^T r_hat becomes the reference of loop j-1
      float acc[kTok];
#pragma unroll
      for (int t = 0; t < kTok; ++t) acc[t] = 0.f;
      if (hadamard) {   // R^T = R; x_s is free (this loop's residual is no longer read)
#pragma unroll
        for (int t = 0; t < kTok; ++t) acc[t] = u_s[t][tid];
        hadamard128<kTok>(acc, tid, &x_s[0][0]);
      } else if (act) {
        for (int k = 0; k < d; ++k) {
          float r = __ldg(a.R + (size_t)k * d + tid);
#pragma unroll
          for (int t = 0; t < kTok; ++t) acc[t] = fmaf(r, u_s[t][k], acc[t]);
        }
      }
      __syncthreads();   // everyone has read ref_s / u_s of this loop
      if (act) {
#pragma unroll
        for (int t = 0; t < kTok; ++t) ref_s[t][tid] = fmaf(cb_s[t], ref_s[t][tid], acc[t]);
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_append(const rq_cache& c, int layer, int group, int batch,
                          const __nv_bfloat16* kv, const int32_t* seq_lens, int n_tokens,
                          int32_t* status, cudaStream_t stream) {
  AppendArgs a;
  a.g = c.geom;
  a.base = c.base;
  a.R = c.R;
  a.kv = kv;
  a.seq_lens = seq_lens;
  a.status = status;
  a.layer = layer;
  a.group = group;
  a.batch = batch;
  a.n = n_tokens;
  // aligned 16-position blocks touched by n tokens starting anywhere: at most ceil(n/16) + 1;
  // a short append in shared mode takes one CTA per (K/V, residual loop)
  const bool split = !(c.geom.mode & RQ_MODE_CHAINED) && c.geom.P > 1 && n_tokens <= kTok;
  if ((int64_t)batch * c.geom.H > 65535) return cudaErrorNotSupported;   // grid.y holds (row, head)
  dim3 grid((n_tokens + kTok - 1) / kTok + 1, batch * c.geom.H, split ? 2 * (c.geom.P - 1) : 2);
  if (c.geom.d == 128) return launch_dependent(append_kernel<128>, grid, dim3(kThreads), 0, stream, a);
  if (c.geom.d == 96) return launch_dependent(append_kernel<96>, grid, dim3(kThreads), 0, stream, a);
  return cudaErrorNotSupported;
}

}  // namespace rq

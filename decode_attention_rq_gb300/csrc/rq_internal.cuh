// Internal declarations shared by the librq translation units (not installed).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rq.h"

namespace rq {

constexpr int kTile = 64;            // token slots per tile (layout constant, see rq.h)
constexpr int kAnchorBits = 4;
constexpr int kResBits = 2;
constexpr int kMaxLoops = 16;      // loops per anchor group (Huginn-shaped groups of up to 16)
constexpr int kStatusWords = 4;      // int32 status word at the start of a workspace
constexpr unsigned long long kWaitNs = 2000000000ull;  // give up an mbarrier wait after 2 s

// Byte geometry of a cache (mirrors the layout statement in rq.h).
struct Geom {
  int L, P, G, H, d, g, ng, Bmax, Nmax, ntiles, mode;
  int Hq, qpk;                                      // query heads; query heads per KV head
  int64_t a_codes, r_codes, meta, a_tile, r_tile;   // per tile, bytes
  int64_t plane_a, plane_r, region;                 // bytes
  // paged layout (rq_cache_create_paged): tile t of row b is page table[b * max_tiles + t]
  // of the (layer, group)'s pool; a page holds that tile of every plane of every head
  int paged, num_pages, max_tiles;
  const int32_t* table;                             // device
  int64_t head_block, page_bytes;                   // one head's tiles of all planes; H of them

  __host__ __device__ int64_t region_offset(int layer, int group, int b, int h) const {
    return ((((int64_t)layer * G + group) * Bmax + b) * H + h) * region;
  }
  __host__ __device__ int64_t anchor_plane(int kv) const { return (int64_t)kv * plane_a; }
  __host__ __device__ int64_t res_plane(int j, int kv) const {
    return 2 * plane_a + (int64_t)(2 * j + kv) * plane_r;
  }
  // Byte offset of tile t of one plane (anchor, or residual plane j; kv 0 = K, 1 = V)
  // of (layer, group, row b, head h); `page` is that tile's page in the paged layout.
  __host__ __device__ int64_t tile_offset(int layer, int group, int b, int h, bool anchor, int j, int kv, int t,
                                          int page) const {
    if (paged)
      return (((int64_t)layer * G + group) * num_pages + page) * page_bytes + (int64_t)h * head_block +
             (anchor ? (int64_t)kv * a_tile : 2 * a_tile + (int64_t)(2 * j + kv) * r_tile);
    return region_offset(layer, group, b, h) + (anchor ? anchor_plane(kv) : res_plane(j, kv)) +
           (int64_t)t * (anchor ? a_tile : r_tile);
  }
};

// Returns false when the shape is outside the supported set.
bool make_geom(const rq_config& c, Geom* g);

}  // namespace rq

struct rq_cache {
  rq_config cfg;
  rq::Geom geom;
  uint8_t* base;
  const float* R;
  int device;
  int num_sms;
};

namespace rq {

// Device ordinals the launchers keep per-device state for (kernel attributes,
// the no-allocation workspace address).
constexpr int kMaxDevices = 64;

// True when the device current on the calling thread is the one the cache was
// created on: the cache's memory, R and the caller's tensors live there, and a
// kernel launched on another device would read addresses it cannot map.
inline bool on_cache_device(const rq_cache& c) {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == c.device;
}

// ---- launchers (one per translation unit) ----
cudaError_t launch_append(const rq_cache& c, int layer, int group, int batch,
                          const __nv_bfloat16* kv, const int32_t* seq_lens, int n_tokens,
                          int32_t* status, cudaStream_t stream);

size_t decode_workspace_bytes(const Geom& g, int batch, int num_sms);
int decode_max_chained_loops();   // chained-mode decode reads at most this many loops' planes
// kv_all (anchor loop only, else ignored): [P][2][batch][H][d] current token of
// every loop, compressed into the cache at seq_lens[b] by the call's merge kernel
cudaError_t launch_decode(const rq_cache& c, int layer, int group, int loop, int batch,
                          const __nv_bfloat16* q, const __nv_bfloat16* k_cur,
                          const __nv_bfloat16* v_cur, const int32_t* seq_lens, float scale,
                          float* out, void* workspace, cudaStream_t stream,
                          const __nv_bfloat16* kv_all = nullptr);

size_t bf16_workspace_bytes(int batch, int heads, int d, int num_sms);
cudaError_t launch_bf16(const __nv_bfloat16* k, const __nv_bfloat16* v,
                        const __nv_bfloat16* k_cur, const __nv_bfloat16* v_cur,
                        const __nv_bfloat16* q, const int32_t* seq_lens, int batch, int heads,
                        int d, int max_seq, float scale, float* out, void* workspace,
                        int num_sms, cudaStream_t stream);

// ---- device helpers: shared-memory TMA bulk copies and mbarriers ----
#if defined(__CUDACC__)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// try_wait that lets the hardware suspend the thread (up to about a millisecond)
// until the phase completes, instead of spinning on issue slots
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity; gives up after kWaitNs of wall time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity))
    if (global_ns() - t0 > kWaitNs) return false;
  return true;
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// L2 policy for data read once (the cache stream): evicted first, so that small
// reused data (the rotation, query packs, partials) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// 4-byte asynchronous global -> shared copy (no register holds the value; the
// issuing thread waits for its copies with cp_async_wait_all before reading them).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}
// Two E4M3 bytes (low byte first) -> two floats, exact.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t v) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tmov.b16 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "h"(v));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hh);
}
// 2^x by the SFU's approximation (relative error about 2^-22; results below the
// normal range flush to 0; 2^-inf = 0): the softmax weights of the streaming
// loops, which are then rounded to 16-bit fixed point or summed in float32.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Walsh-Hadamard rotation (RQ_MODE_HADAMARD, d = 128): u = H v / sqrt(128) for
// NT vectors whose channels are held one per thread (thread i < 128 holds
// channel i of each).  Butterfly stages h = 1, 2, ..., 64 turn every pair
// (a, b) = (v[j], v[j + h]), j & h == 0, into (a + b, a - b), each rounded to
// binary32 -- stages below 32 across lanes, 32 and 64 through xs ([NT][128]
// floats of shared memory) -- then one binary32 product with the binary32 value
// of 1/sqrt(128).  H is symmetric: the same call applies R^T.  It holds
// barriers: every thread of the CTA calls it; threads >= 128 only take part
// in those (their values are not used).
constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;
template <int NT>
__device__ __forceinline__ void hadamard128(float (&v)[NT], int i, float* xs) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float p = __shfl_xor_sync(0xffffffffu, v[t], h);
      v[t] = (i & h) ? __fsub_rn(p, v[t]) : __fadd_rn(v[t], p);
    }
  }
#pragma unroll
  for (int h = 32; h < 128; h <<= 1) {
    if (i < 128) {
#pragma unroll
      for (int t = 0; t < NT; ++t) xs[t * 128 + i] = v[t];
    }
    __syncthreads();
    float p[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) p[t] = i < 128 ? xs[t * 128 + (i ^ h)] : 0.f;
    __syncthreads();
#pragma unroll
    for (int t = 0; t < NT; ++t) v[t] = (i & h) ? __fsub_rn(p[t], v[t]) : __fadd_rn(v[t], p[t]);
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) v[t] = __fmul_rn(v[t], kInvSqrt128);
}
// Page of tile t of row b (paged layout) from a raw block-table entry.  An entry
// outside [0, num_pages) sets status[2] and gives -1 (the caller skips the tile
// or reads page 0 instead: nothing outside the pool is touched).
__device__ __forceinline__ int checked_page(const Geom& g, int raw, int32_t* status) {
  if (raw >= 0 && raw < g.num_pages) return raw;
  if (status) atomicExch(&status[2], 1);
  return -1;
}
__device__ __forceinline__ int raw_page(const Geom& g, int b, int t) {
  return __ldg(g.table + (size_t)b * g.max_tiles + t);
}
// Programmatic dependent launch: let the next kernel of the stream start its
// prologue; wait until the kernel before this one has finished and its writes
// are visible (returns at once when launched without the dependency).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// Launch with programmatic stream serialization: the kernel may start before the
// previous kernel on the stream finishes and must call pdl_wait() before it reads
// anything that kernel (or earlier work) produced.
template <typename... Args>
cudaError_t launch_dependent(void (*k)(Args...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace rq

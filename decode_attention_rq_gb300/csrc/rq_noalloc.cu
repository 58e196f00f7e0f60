// rq_decode_attention_noalloc: rq_decode_attention with its scratch memory
// built into the library, for callers that cannot allocate device memory.
//
// The paper has no counterpart to this entry point; it exists for callers of
// this library that are handed their buffers and may not allocate more:
// plugins whose host application owns all device memory, code that runs
// under a fixed memory budget reserved up front, or code on a path where an
// allocation could block or fail.  Such a caller still passes the inputs and
// the output; the split-K workspace (status word, per-CTA partial softmax
// states, query packs) lives in one file-scope device
// array of RQ_NOALLOC_WORKSPACE_BYTES.  Every device on which this library is
// loaded holds that array until the process exits.
//
// The array's name in host code is only a host-side handle for the symbol,
// not a device address: a kernel given it would fault, or on a system where
// the GPU can reach host memory, silently touch the wrong memory.  Its device
// address is therefore looked up with cudaGetSymbolAddress, once per device,
// on the first call made with that device current, and passed to the kernel.
//
// Every call shares the array and finds in it what the last call left.  A
// call clears the part it uses (the status word must start at zero) on its
// own stream before launching, so calls that overlap on the
// GPU -- two streams, or two threads -- race on the array and give wrong
// results: serialize them.
#include <mutex>

#include "rq_internal.cuh"

// Workspace of every rq_decode_attention_noalloc call (zero-initialised at load).
static __device__ __align__(256) uint8_t g_noalloc_workspace[RQ_NOALLOC_WORKSPACE_BYTES];

namespace rq {
namespace {

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices];   // device address of the array, per device ordinal

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of g_noalloc_workspace on the current device; looked up once.
cudaError_t noalloc_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace rq

using namespace rq;

extern "C" rq_status rq_decode_attention_noalloc(rq_cache* cache, int32_t layer, int32_t group,
                                                 int32_t loop, int32_t batch, const void* q,
                                                 const void* k_cur, const void* v_cur,
                                                 const int32_t* seq_lens, float softmax_scale,
                                                 float* out, int32_t* status, void* stream) {
  if (!cache || !q || !k_cur || !v_cur || !seq_lens || !out) return RQ_ERR_INVALID_ARG;
  if (!on_cache_device(*cache)) return RQ_ERR_INVALID_ARG;
  const Geom& g = cache->geom;
  if (layer < 0 || layer >= g.L || group < 0 || group >= g.G || loop < 0 || loop >= g.P ||
      batch <= 0)
    return RQ_ERR_INVALID_ARG;
  if (batch > g.Bmax) return RQ_ERR_CAPACITY;
  if (batch > RQ_MAX_DECODE_BATCH) return RQ_ERR_UNSUPPORTED;
  if ((g.mode & RQ_MODE_CHAINED) && g.P > decode_max_chained_loops()) return RQ_ERR_UNSUPPORTED;
  const size_t need = decode_workspace_bytes(g, batch, cache->num_sms);
  if (need > (size_t)RQ_NOALLOC_WORKSPACE_BYTES) return RQ_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k_cur) || !aligned16(v_cur) || !aligned16(seq_lens) ||
      !aligned16(out) || (status && !aligned16(status)))
    return RQ_ERR_ALIGNMENT;
  void* ws = nullptr;
  if (noalloc_workspace(&ws) != cudaSuccess) return RQ_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word must start at zero; clearing the whole extent this call uses
  // also drops whatever an earlier, aborted call left behind
  if (cudaMemsetAsync(ws, 0, need, st) != cudaSuccess) return RQ_ERR_CUDA;
  cudaError_t e = launch_decode(*cache, layer, group, loop, batch,
                                static_cast<const __nv_bfloat16*>(q),
                                static_cast<const __nv_bfloat16*>(k_cur),
                                static_cast<const __nv_bfloat16*>(v_cur), seq_lens, softmax_scale,
                                out, ws, st);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? RQ_ERR_UNSUPPORTED : RQ_ERR_CUDA;
  // the status word sits in the array's first 16 bytes; hand it to the caller if asked
  if (status && cudaMemcpyAsync(status, ws, 16, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return RQ_ERR_CUDA;
  return RQ_OK;
}

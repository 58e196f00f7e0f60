// C-ABI entry points of librq: argument checks, geometry, dispatch to the kernels.
#include <cstdlib>
#include <new>

#include "rq_internal.cuh"

namespace rq {

bool make_geom(const rq_config& c, Geom* g) {
  if (c.num_layers <= 0 || c.num_groups <= 0 || c.num_heads <= 0 || c.max_batch <= 0 ||
      c.max_seq_len <= 0)
    return false;
  if (c.loops_per_group < 1 || c.loops_per_group > kMaxLoops) return false;
  if (c.head_dim != 96 && c.head_dim != 128) return false;
  if (c.group_size != 16 && c.group_size != 32) return false;
  if (c.head_dim % c.group_size) return false;
  if (c.mode & ~(RQ_MODE_CHAINED | RQ_MODE_NORM_RATIO | RQ_MODE_HADAMARD)) return false;
  if ((c.mode & RQ_MODE_HADAMARD) && c.head_dim != 128) return false;   // a power of two
  g->L = c.num_layers;
  g->P = c.loops_per_group;
  g->G = c.num_groups;
  g->H = c.num_heads;
  if (c.num_query_heads < 0 || (c.num_query_heads > 0 && c.num_query_heads % c.num_heads)) return false;
  g->Hq = c.num_query_heads > 0 ? c.num_query_heads : c.num_heads;
  g->qpk = g->Hq / g->H;
  g->d = c.head_dim;
  g->g = c.group_size;
  g->ng = c.head_dim / c.group_size;
  g->Bmax = c.max_batch;
  g->Nmax = c.max_seq_len;
  g->mode = c.mode;
  g->ntiles = (c.max_seq_len + kTile - 1) / kTile;
  g->a_codes = (int64_t)kTile * g->d / 2;
  g->r_codes = (int64_t)kTile * g->d / 4;
  g->meta = (int64_t)kTile * g->ng * 2;
  g->a_tile = g->a_codes + g->meta;
  g->r_tile = g->r_codes + g->meta + (int64_t)kTile * 2;
  g->plane_a = (int64_t)g->ntiles * g->a_tile;
  g->plane_r = (int64_t)g->ntiles * g->r_tile;
  g->region = 2 * g->plane_a + 2 * (int64_t)(g->P - 1) * g->plane_r;
  g->paged = 0;
  g->num_pages = 0;
  g->max_tiles = g->ntiles;
  g->table = nullptr;
  g->head_block = 2 * g->a_tile + 2 * (int64_t)(g->P - 1) * g->r_tile;
  g->page_bytes = (int64_t)g->H * g->head_block;
  return true;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int current_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace rq

using namespace rq;

extern "C" {

size_t rq_cache_bytes(const rq_config* cfg) {
  Geom g;
  if (!cfg || !make_geom(*cfg, &g)) return 0;
  return (size_t)g.L * g.G * g.Bmax * g.H * (size_t)g.region;
}

rq_status rq_cache_create(const rq_config* cfg, void* dev_buf, size_t bytes, const float* R_dev,
                          rq_cache** out) {
  if (!cfg || !dev_buf || !out) return RQ_ERR_INVALID_ARG;
  const bool hadamard = (cfg->mode & RQ_MODE_HADAMARD) != 0;
  if (!R_dev && !hadamard) return RQ_ERR_INVALID_ARG;
  Geom g;
  if (!make_geom(*cfg, &g)) return RQ_ERR_UNSUPPORTED;
  if (bytes < rq_cache_bytes(cfg)) return RQ_ERR_CAPACITY;
  if (!aligned16(dev_buf) || (R_dev && !aligned16(R_dev))) return RQ_ERR_ALIGNMENT;
  rq_cache* c = new (std::nothrow) rq_cache;
  if (!c) return RQ_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->geom = g;
  c->base = static_cast<uint8_t*>(dev_buf);
  c->R = R_dev;
  c->device = 0;
  cudaGetDevice(&c->device);
  c->num_sms = current_sms();
  if (c->num_sms <= 0) {
    delete c;
    return RQ_ERR_CUDA;
  }
  *out = c;
  return RQ_OK;
}

size_t rq_cache_paged_bytes(const rq_config* cfg, int32_t num_pages) {
  Geom g;
  if (!cfg || !make_geom(*cfg, &g) || num_pages <= 0) return 0;
  return (size_t)g.L * g.G * (size_t)num_pages * (size_t)g.page_bytes;
}

rq_status rq_cache_create_paged(const rq_config* cfg, int32_t num_pages, void* dev_pool, size_t bytes,
                                const int32_t* block_table, int32_t max_tiles_per_row, const float* R_dev,
                                rq_cache** out) {
  if (!cfg || !dev_pool || !block_table || !out) return RQ_ERR_INVALID_ARG;
  const bool hadamard = (cfg->mode & RQ_MODE_HADAMARD) != 0;
  if (!R_dev && !hadamard) return RQ_ERR_INVALID_ARG;
  Geom g;
  if (!make_geom(*cfg, &g)) return RQ_ERR_UNSUPPORTED;
  if (num_pages <= 0 || max_tiles_per_row < g.ntiles) return RQ_ERR_INVALID_ARG;
  if (bytes < rq_cache_paged_bytes(cfg, num_pages)) return RQ_ERR_CAPACITY;
  if (!aligned16(dev_pool) || !aligned16(block_table) || (R_dev && !aligned16(R_dev))) return RQ_ERR_ALIGNMENT;
  g.paged = 1;
  g.num_pages = num_pages;
  g.max_tiles = max_tiles_per_row;
  g.table = block_table;
  rq_cache* c = new (std::nothrow) rq_cache;
  if (!c) return RQ_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->geom = g;
  c->base = static_cast<uint8_t*>(dev_pool);
  c->R = R_dev;
  c->device = 0;
  cudaGetDevice(&c->device);
  c->num_sms = current_sms();
  if (c->num_sms <= 0) {
    delete c;
    return RQ_ERR_CUDA;
  }
  *out = c;
  return RQ_OK;
}

rq_status rq_cache_destroy(rq_cache* cache) {
  delete cache;
  return RQ_OK;
}

rq_status rq_append(rq_cache* cache, int32_t layer, int32_t group, int32_t batch, const void* kv,
                    const int32_t* seq_lens, int32_t n_tokens, int32_t* status, void* stream) {
  if (!cache || !kv || !seq_lens) return RQ_ERR_INVALID_ARG;
  if (!on_cache_device(*cache)) return RQ_ERR_INVALID_ARG;
  const Geom& g = cache->geom;
  if (layer < 0 || layer >= g.L || group < 0 || group >= g.G || batch <= 0 || n_tokens < 0)
    return RQ_ERR_INVALID_ARG;
  if (batch > g.Bmax || n_tokens > g.Nmax) return RQ_ERR_CAPACITY;
  if (!aligned16(kv) || !aligned16(seq_lens) || (status && !aligned16(status)))
    return RQ_ERR_ALIGNMENT;
  if (n_tokens == 0) return RQ_OK;
  cudaError_t e = launch_append(*cache, layer, group, batch, static_cast<const __nv_bfloat16*>(kv),
                                seq_lens, n_tokens, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RQ_OK : (e == cudaErrorNotSupported ? RQ_ERR_UNSUPPORTED : RQ_ERR_CUDA);
}

size_t rq_decode_workspace_bytes(const rq_config* cfg, int32_t batch) {
  Geom g;
  if (!cfg || !make_geom(*cfg, &g) || batch <= 0) return 0;
  return decode_workspace_bytes(g, batch, current_sms());
}

rq_status rq_decode_attention(rq_cache* cache, int32_t layer, int32_t group, int32_t loop,
                              int32_t batch, const void* q, const void* k_cur, const void* v_cur,
                              const int32_t* seq_lens, float softmax_scale, float* out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (!cache || !q || !k_cur || !v_cur || !seq_lens || !out || !workspace)
    return RQ_ERR_INVALID_ARG;
  if (!on_cache_device(*cache)) return RQ_ERR_INVALID_ARG;
  const Geom& g = cache->geom;
  if (layer < 0 || layer >= g.L || group < 0 || group >= g.G || loop < 0 || loop >= g.P ||
      batch <= 0)
    return RQ_ERR_INVALID_ARG;
  if (batch > g.Bmax) return RQ_ERR_CAPACITY;
  if (batch > RQ_MAX_DECODE_BATCH) return RQ_ERR_UNSUPPORTED;
  if ((g.mode & RQ_MODE_CHAINED) && g.P > decode_max_chained_loops()) return RQ_ERR_UNSUPPORTED;
  if (workspace_bytes < decode_workspace_bytes(g, batch, cache->num_sms)) return RQ_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k_cur) || !aligned16(v_cur) || !aligned16(seq_lens) ||
      !aligned16(out) || !aligned16(workspace))
    return RQ_ERR_ALIGNMENT;
  cudaError_t e = launch_decode(*cache, layer, group, loop, batch,
                                static_cast<const __nv_bfloat16*>(q),
                                static_cast<const __nv_bfloat16*>(k_cur),
                                static_cast<const __nv_bfloat16*>(v_cur), seq_lens, softmax_scale,
                                out, workspace, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RQ_OK : (e == cudaErrorNotSupported ? RQ_ERR_UNSUPPORTED : RQ_ERR_CUDA);
}

rq_status rq_decode_attention_append(rq_cache* cache, int32_t layer, int32_t group, int32_t batch,
                                     const void* q, const void* kv_cur, const int32_t* seq_lens,
                                     float softmax_scale, float* out, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (!cache || !q || !kv_cur || !seq_lens || !out || !workspace) return RQ_ERR_INVALID_ARG;
  if (!on_cache_device(*cache)) return RQ_ERR_INVALID_ARG;
  const Geom& g = cache->geom;
  if (layer < 0 || layer >= g.L || group < 0 || group >= g.G || batch <= 0) return RQ_ERR_INVALID_ARG;
  if (batch > g.Bmax) return RQ_ERR_CAPACITY;
  if (batch > RQ_MAX_DECODE_BATCH) return RQ_ERR_UNSUPPORTED;
  if ((g.mode & RQ_MODE_CHAINED) && g.P > decode_max_chained_loops()) return RQ_ERR_UNSUPPORTED;
  if (workspace_bytes < decode_workspace_bytes(g, batch, cache->num_sms)) return RQ_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(kv_cur) || !aligned16(seq_lens) || !aligned16(out) ||
      !aligned16(workspace))
    return RQ_ERR_ALIGNMENT;
  // the anchor loop's K and V of the current token: blocks (P-1, 0) and (P-1, 1) of kv_cur
  const auto* kv = static_cast<const __nv_bfloat16*>(kv_cur);
  const size_t block = (size_t)batch * g.H * g.d;
  const __nv_bfloat16* k_cur = kv + (size_t)(2 * (g.P - 1)) * block;
  cudaError_t e = launch_decode(*cache, layer, group, g.P - 1, batch, static_cast<const __nv_bfloat16*>(q),
                                k_cur, k_cur + block, seq_lens, softmax_scale, out, workspace,
                                static_cast<cudaStream_t>(stream), kv);
  return e == cudaSuccess ? RQ_OK : (e == cudaErrorNotSupported ? RQ_ERR_UNSUPPORTED : RQ_ERR_CUDA);
}

size_t rq_bf16_workspace_bytes(int32_t batch, int32_t num_heads, int32_t head_dim) {
  if (batch <= 0 || num_heads <= 0 || (head_dim != 96 && head_dim != 128)) return 0;
  return bf16_workspace_bytes(batch, num_heads, head_dim, current_sms());
}

rq_status rq_decode_attention_bf16(const void* k_cache, const void* v_cache, const void* k_cur,
                                   const void* v_cur, const void* q, const int32_t* seq_lens,
                                   int32_t batch, int32_t num_heads, int32_t head_dim,
                                   int32_t max_seq, float softmax_scale, float* out,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!k_cache || !v_cache || !k_cur || !v_cur || !q || !seq_lens || !out || !workspace)
    return RQ_ERR_INVALID_ARG;
  if (batch <= 0 || num_heads <= 0 || max_seq <= 0) return RQ_ERR_INVALID_ARG;
  if (batch > RQ_MAX_DECODE_BATCH) return RQ_ERR_UNSUPPORTED;
  if (head_dim != 96 && head_dim != 128) return RQ_ERR_UNSUPPORTED;
  int sms = current_sms();
  if (sms <= 0) return RQ_ERR_CUDA;
  if (workspace_bytes < bf16_workspace_bytes(batch, num_heads, head_dim, sms))
    return RQ_ERR_WORKSPACE;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_cur) || !aligned16(v_cur) ||
      !aligned16(q) || !aligned16(seq_lens) || !aligned16(out) || !aligned16(workspace))
    return RQ_ERR_ALIGNMENT;
  cudaError_t e = launch_bf16(
      static_cast<const __nv_bfloat16*>(k_cache), static_cast<const __nv_bfloat16*>(v_cache),
      static_cast<const __nv_bfloat16*>(k_cur), static_cast<const __nv_bfloat16*>(v_cur),
      static_cast<const __nv_bfloat16*>(q), seq_lens, batch, num_heads, head_dim, max_seq,
      softmax_scale, out, workspace, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

const char* rq_status_string(rq_status s) {
  switch (s) {
    case RQ_OK: return "ok";
    case RQ_ERR_INVALID_ARG: return "invalid argument";
    case RQ_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case RQ_ERR_CAPACITY: return "capacity exceeded (batch or sequence length)";
    case RQ_ERR_WORKSPACE: return "workspace too small";
    case RQ_ERR_CUDA: return "CUDA error";
    case RQ_ERR_UNSUPPORTED: return "unsupported shape";
    case RQ_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

}  // extern "C"

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
//   * Three kernels per call.  qprep_kernel (one CTA per (row, head)) applies
//     R to the query and turns q and R q into the f16 operand images the
//     scoring products use.  decode_kernel streams the cache and writes one partial
//     softmax state per (CTA, segment).  merge_kernel (one CTA per (row,
//     head)) combines the partials, adds the current BF16 token, applies R^T
//     once and writes the output.  All three are launched as programmatic
//     dependents of the kernel before them: what needs only the call's inputs
//     (the prep's whole query pack; the decode kernel's work split and first
//     cache copies; the merge's R in shared memory and current token) overlaps
//     that kernel, and each waits for it (griddepcontrol.wait) only before
//     reading what it wrote or writing what it may still read.
//   * Work units are (row, head, 128 tokens).  A fixed grid of
//     num_SMs x (CTAs resident per SM) takes equal contiguous ranges of the flattened
//     unit list (ranges cross (row, head) boundaries), so every SM streams
//     the same number of tiles whatever the batch and lengths.
//   * A unit's plane slices (anchor K/V, the residual K/V planes this loop
//     reads) are contiguous and 16-byte aligned: one thread issues 1-D TMA
//     bulk copies into a shared-memory ring tracked by mbarriers (bounded
//     waits).  Contiguous cache: a stage holds each plane's two tiles
//     together, one copy per plane; paged cache: tile by tile, two copies per
//     tile (the anchor pair, the residual planes read), neighbours in the
//     tile's page.  Fewer copies matter: the issuing thread, also a consumer,
//     stalls while the SM's copy engine is busy.
//   * Scores use the rotated query: q.(c a_hat + R^T r_hat) = c (q.a_hat) +
//     (R q).r_hat.  The value side accumulates the anchor part and the
//     rotated residual part apart; R^T is applied once, in the merge.
//   * Per group, q.x_hat = s * sum(q * code) + o * sum(q), and the value side
//     keeps the offsets as one scalar per (unit, group): the work per code is
//     one multiply-add against a small integer.
//   * Those multiply-adds are f16 tensor-core products (mma.sync m16n8k16,
//     f32 accumulation).  A code word masked with 0x000F000F, 0x00F000F0 or
//     0x00030003 << 2m (after a shift by 8 for the other two bytes) is an f16
//     pair whose bit patterns are small integers: values code * 2^-24 (times
//     16 or 4^m), exact, with no conversion and no bias.  Scoring: tokens x
//     channels against the query (q, and R q for the residual planes) split
//     into two f16 pieces (about 22 bits) in the B operand, one column pair
//     per channel group, so each lane's accumulator holds one group's dot
//     products.  Values: channels x tokens against the softmax-times-scale
//     weights of the unit, again two f16 pieces per weight, so every weight
//     keeps its own relative precision (no fixed point relative to the
//     unit's largest weight: a softmax that one key dominates loses nothing).
//     The 16 / 4^m factors of the masked codes are divided out of the B
//     operands.  The tokens of a lane's two score rows (t, t + 2) are the
//     pair one B register of the value products holds.
//   * Online softmax in base 2 (scale * log2(e) folded into q).
//   * Variants: grouped-query attention runs the multi-query kernel
//     (rq_decode_gqa.cu: a unit is (row, head group, 128 tokens), the tiles
//     staged once for 2 or 4 query heads) for calls reading at most one
//     residual plane, and per query head otherwise;
//     the paged layout (decode_kernel<..., PAGED>) takes each tile's address
//     from the block table, fetched one unit ahead by the producer thread;
//     the Walsh-Hadamard mode replaces R q and R^T acc by the fast transform;
//     the anchor-loop call can also append the current token in its merge
//     kernel (rq_token_append.cuh).  Every kernel asks for the largest
//     shared-memory carveout so that each can start beside the one before it.
#include "rq_decode_kernels.cuh"

namespace rq {
namespace {

template <int D, int GS, bool PAGED>
cudaError_t launch_p(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  switch (nres) {
    case 0: return launch_t<D, GS, 0, PAGED>(a, num_sms, stream);
    case 1: return launch_t<D, GS, 1, PAGED>(a, num_sms, stream);
    case 2: return launch_t<D, GS, 2, PAGED>(a, num_sms, stream);
    case 3: return launch_t<D, GS, 3, PAGED>(a, num_sms, stream);
  }
  return launch_decode_long_chain(a, num_sms, nres, stream);   // 4 .. 7 planes
}

template <int D, int GS>
cudaError_t launch_d(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  return a.g.paged ? launch_p<D, GS, true>(a, num_sms, nres, stream) : launch_p<D, GS, false>(a, num_sms, nres, stream);
}

int pstride_for(int d) { return ((2 + 2 * d) + 3) / 4 * 4; }

}  // namespace

int decode_max_chained_loops() { return kMaxRes + 1; }

// Query heads per work unit: grouped-query caches take the heads of a KV head in
// groups of 4 (or 2) through the multi-query kernel (rq_decode_gqa.cu).
static int decode_qh(const Geom& g) { return g.qpk % 4 == 0 ? 4 : (g.qpk % 2 == 0 ? 2 : 1); }

// Partial rows: the per-head kernel writes row cta + bh (at most 3 CTAs per SM);
// the multi-query kernel row (cta + group) * qh + h (at most 2 CTAs per SM).
static size_t partials_bytes(const Geom& g, int batch, int num_sms) {
  const int qh = decode_qh(g);
  const size_t C = (size_t)num_sms * (kMaxCtasPerSm > 2 * qh ? kMaxCtasPerSm : 2 * qh), bh = (size_t)batch * g.Hq;
  return ((C + bh) * pstride_for(g.d) * sizeof(float) + 255) / 256 * 256;
}

// Workspace: status word (256 B slot) | partials (C + batch*Hq) x pstride floats | query packs.
size_t decode_workspace_bytes(const Geom& g, int batch, int num_sms) {
  const size_t bh = (size_t)batch * g.Hq;
  return 256 + partials_bytes(g, batch, num_sms) + bh * kPackWords * sizeof(uint32_t);
}

cudaError_t launch_decode(const rq_cache& c, int layer, int group, int loop, int batch,
                          const __nv_bfloat16* q, const __nv_bfloat16* k_cur,
                          const __nv_bfloat16* v_cur, const int32_t* seq_lens, float scale,
                          float* out, void* workspace, cudaStream_t stream,
                          const __nv_bfloat16* kv_all) {
  if (batch > kMaxRows) return cudaErrorInvalidValue;
  const int P = c.geom.P;
  const bool chained = (c.geom.mode & RQ_MODE_CHAINED) != 0;
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
  a.kv_all = loop == P - 1 ? kv_all : nullptr;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<int32_t*>(ws);
  a.partials = reinterpret_cast<float*>(ws + 256);
  a.packs = reinterpret_cast<uint32_t*>(ws + 256 + partials_bytes(c.geom, batch, c.num_sms));
  a.pstride = pstride_for(c.geom.d);
  a.layer = layer;
  a.group = group;
  a.batch = batch;
  a.res0 = loop;
  a.qh = 1;
  a.qscale = scale * kLog2e;
  const int d = c.geom.d, gs = c.geom.g, n = c.num_sms;
  // grouped-query attention: the query heads of a KV head in groups of 4 (or 2)
  // per pass over its tiles
  const int qh = decode_qh(c.geom);
  if (qh > 1 && nres <= 1) {
    a.qh = qh;
    return launch_decode_gqa(a, n, nres, stream);
  }
  if (d == 128 && gs == 32) return launch_d<128, 32>(a, n, nres, stream);
  if (d == 128 && gs == 16) return launch_d<128, 16>(a, n, nres, stream);
  if (d == 96 && gs == 32) return launch_d<96, 32>(a, n, nres, stream);
  if (d == 96 && gs == 16) return launch_d<96, 16>(a, n, nres, stream);
  return cudaErrorNotSupported;
}

}  // namespace rq

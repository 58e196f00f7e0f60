/*
 * rq.h - ResidualQuant KV cache and decode attention for NVIDIA GB300 (sm_103a).
 *
 * ResidualQuant (the learnaivisually explainer "ResidualQuant stores
 * looped-Transformer KV caches as 2-bit residuals", and the ai4snews summary
 * of the arXiv paper) compresses the KV cache of a looped Transformer.  The
 * last loop of each loop group is stored as an INT4 "anchor"; every earlier
 * loop l is stored as a 2-bit code of the rotated residual
 *     u_l = R (kv_l - c_l * anchor_hat),  c_l = <kv_l, anchor_hat> / <anchor_hat, anchor_hat>,
 * with c_l kept in BF16 and R a fixed orthogonal rotation.  Channels are
 * grouped (g = 32 or 16) with an FP8-E4M3 scale and offset per group.
 * Decode attention rebuilds c * anchor_hat + R^T dequant(u) on chip and never
 * writes the rebuilt K/V to memory.
 *
 * Conventions for every entry point
 *   - Device pointers are caller-owned device memory (e.g. from PyTorch);
 *     the library never allocates or frees device memory and never
 *     synchronizes the device.  Host pointers are marked "host".
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it.  The decode calls
 *     launch their kernels as programmatic dependents of the work before
 *     them on the stream, and those kernels read their inputs (queries,
 *     current K/V, seq_lens, cache) before waiting for it.  A kernel that
 *     does not release its dependents early (no griddepcontrol.launch_
 *     dependents) has completed before a call starts, so any such kernel may
 *     write the inputs; a kernel that does release early must not be the one
 *     that writes them (its writes are visible only to a kernel that has
 *     waited for it).
 *   - Argument errors are found on the host before anything is enqueued and
 *     return a status; nothing is launched then.  A failed launch returns
 *     RQ_ERR_CUDA.  Faults inside a kernel surface on a later CUDA call.
 *   - Device pointers must be 16-byte aligned (RQ_ERR_ALIGNMENT).
 *   - A cache belongs to the device that was current when it was created;
 *     a call on it made with another device current returns
 *     RQ_ERR_INVALID_ARG (its memory is not addressable from there).
 *   - Supported shapes: head_dim in {96, 128}; group_size in {16, 32} dividing
 *     head_dim; loops_per_group in [1, 16]; num_query_heads a multiple of
 *     num_heads.  Others: RQ_ERR_UNSUPPORTED.
 *
 * Entry points: rq_cache_bytes / rq_cache_create (contiguous layout) or
 * rq_cache_paged_bytes / rq_cache_create_paged (block-table layout);
 * rq_append (compress new tokens: prefill, or one decode token);
 * rq_decode_workspace_bytes, rq_decode_attention (one loop's attention) and
 * rq_decode_attention_append (the anchor loop's attention plus the current
 * token's append); rq_decode_attention_noalloc (scratch inside the library);
 * rq_bf16_workspace_bytes / rq_decode_attention_bf16 (the uncompressed
 * comparator); rq_status_string.
 *
 * ---------------------------------------------------------------------------
 * Cache byte layout (this library's format; the pages fix the record
 * contents, not their placement)
 *   The cache is L x G x max_batch x H regions, index
 *   ((layer * G + group) * max_batch + b) * H + h, each `region` bytes.
 *   A region holds planes AK, AV, then RK_j, RV_j for j = 0 .. P-2.
 *   Each plane is ntiles = ceil(max_seq_len / 64) tiles of 64 token slots;
 *   tile t holds positions 64t .. 64t+63.
 *     anchor tile  (AK, AV)  : codes[64 * d/2] | meta[64 * ng * 2]
 *     residual tile (RK, RV) : codes[64 * d/4] | meta[64 * ng * 2] | c[64 * 2]
 *   K codes are token-major: row r = the token's d codes;
 *     INT4 byte i = ch 2i (bits 0-3) | ch 2i+1 (bits 4-7);
 *     INT2 byte i = ch 4i+m in bits 2m..2m+1.
 *   V codes are channel-major: row ch = that channel's 64 token codes in
 *     32-bit words; INT4 word w (tokens 8w..8w+7): byte i = token 8w+i
 *     (bits 0-3) | token 8w+4+i (bits 4-7); INT2 word j (tokens 16j..16j+15):
 *     byte i holds token 16j+4m+i in bits 2m..2m+1, m = 0..3.  Masking a word
 *     with 0x0F0F0F0F, 0xF0F0F0F0 or 0x03030303 << 2m leaves four consecutive
 *     tokens, one per byte.
 *   meta row r: for each channel group, the E4M3 scale byte then the E4M3
 *     offset byte.  c slot r: BF16, little-endian.
 *   Every tile and sub-block size is a multiple of 16 bytes.
 *
 * Quantizer (both code widths): per group, o = E4M3(min), s = E4M3((max-min)/(2^b-1)),
 * rounded to nearest even and saturating at +-448; code = the nearest grid
 * point o + k*s to the exact value, ties to even k, clamped to [0, 2^b-1];
 * s == 0 gives code 0.  Dequantized value: s * code + o.
 * ---------------------------------------------------------------------------
 */
#ifndef RQ_H_
#define RQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rq_status {
  RQ_OK = 0,
  RQ_ERR_INVALID_ARG = 1,   /* null pointer, index out of range, bad count */
  RQ_ERR_ALIGNMENT = 2,     /* a device pointer is not 16-byte aligned */
  RQ_ERR_CAPACITY = 3,      /* batch > max_batch, or a write past max_seq_len */
  RQ_ERR_WORKSPACE = 4,     /* workspace smaller than the *_workspace_bytes value */
  RQ_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
  RQ_ERR_UNSUPPORTED = 6,   /* head_dim / group_size / loops outside the supported set */
  RQ_ERR_TIMEOUT = 7        /* a device-side wait gave up (reported via the status word) */
} rq_status;

typedef enum rq_mode {
  RQ_MODE_SHARED = 0,   /* every earlier loop coded against the anchor: 2 plane reads per loop */
  RQ_MODE_CHAINED = 1,  /* loop l coded against the rebuilt loop l+1: reads grow with distance */
  RQ_MODE_NORM_RATIO = 2, /* flag, OR'd with one of the above: the stored coefficient is the
                            norm ratio ||kv_l|| / ||ref|| (the scaling the arXiv summary lists
                            beside least squares among its appendix comparisons) instead of
                            the least-squares <kv_l, ref> / <ref, ref>; decode is unchanged */
  RQ_MODE_HADAMARD = 4  /* flag: the rotation is R = H_d / sqrt(d), H_d the Sylvester Hadamard
                           matrix (entry (i, k) = (-1)^popcount(i & k)), applied as a fast
                           Walsh-Hadamard transform (d log d adds) wherever R or R^T acts;
                           head_dim 128 only.  The explainer's related-explainers list points
                           to a 2-bit KV cache built on a Hadamard rotation; the summary's
                           ablation compares rotation methods.  R_dev may then be NULL. */
} rq_mode;

/* Shape of one cache.  The anchor is 4-bit and residuals 2-bit (fixed). */
typedef struct rq_config {
  int32_t num_layers;       /* L: layers of the shared block */
  int32_t loops_per_group;  /* P: loops per anchor group; the last one is the anchor */
  int32_t num_groups;       /* G: loop groups (Ouro-1.4B: 1 group of 4; Huginn-3.5B: 8 of 4) */
  int32_t num_heads;        /* H: KV heads (the cache stores these) */
  int32_t head_dim;         /* d: 96 or 128 */
  int32_t group_size;       /* g: 16 or 32 channels per quantization group */
  int32_t max_batch;        /* rows of the cache */
  int32_t max_seq_len;      /* token capacity per (layer, group, row, head) */
  int32_t mode;             /* rq_mode: SHARED or CHAINED, optionally | NORM_RATIO | HADAMARD */
  int32_t num_query_heads;  /* Hq: query heads; 0 (or H) = multi-head attention, else a multiple
                               of H (grouped-query: query head qh attends with KV head
                               qh / (Hq / H)).  Decode calls take q and out with Hq heads and
                               the current token's K/V with H heads. */
} rq_config;

typedef struct rq_cache rq_cache;   /* opaque host-side handle; holds no device memory */

/* Bytes of device memory a cache of this shape needs (0 if the shape is invalid).
 * Host only; no CUDA call. */
size_t rq_cache_bytes(const rq_config* cfg);

/* Bind a cache to caller memory.
 *   cfg    host; copied.  cfg->mode: RQ_MODE_SHARED or RQ_MODE_CHAINED, optionally
 *          OR'd with RQ_MODE_NORM_RATIO and RQ_MODE_HADAMARD.  In binary32 the
 *          Hadamard transform runs butterfly stages h = 1, 2, ..., d/2, each pair
 *          (j, j+h) becoming (a+b, a-b) rounded, then one product with the
 *          binary32 value of 1/sqrt(d); the stored codes follow that order.
 *   dev_buf device, >= rq_cache_bytes(cfg) bytes, 16-byte aligned.  Its
 *          contents are the cache; the caller zero-fills it before first use
 *          (only needed for byte-exact comparisons: unwritten slots are never read).
 *   R_dev  device float32 [d][d] row-major, the rotation (orthogonal); caller
 *          keeps it alive and unchanged while the cache is used.  Unused (may be
 *          NULL) with RQ_MODE_HADAMARD.
 *   out    host; receives the handle.  Free it with rq_cache_destroy.
 * Errors: INVALID_ARG (null), UNSUPPORTED (shape), CAPACITY (bytes too small),
 * ALIGNMENT. */
rq_status rq_cache_create(const rq_config* cfg, void* dev_buf, size_t bytes,
                          const float* R_dev, rq_cache** out);

/* Paged layout (block table, as a paged serving engine lays out its KV cache).
 * Instead of a contiguous capacity per (layer, group, row, head), each
 * (layer, group) owns a pool of num_pages pages; a page holds one 64-token tile
 * of every plane (anchor K/V, every residual K/V, with their metadata and
 * coefficients, laid out as in the contiguous tile) of every head:
 *   pool(layer, group) = base + (layer * G + group) * num_pages * page_bytes
 *   page p, head h:      pool + p * page_bytes + h * head_block
 *   head_block = 2 * anchor_tile + 2 * (P - 1) * residual_tile, page_bytes = H * head_block
 *   inside a head block: anchor K tile, anchor V tile, then residual plane j's
 *   K and V tiles for j = 0 .. P-2.
 * Tile t (token positions 64t .. 64t+63) of batch row b lives in page
 * block_table[b * max_tiles_per_row + t]; the same table serves every layer and
 * group.  The caller assigns pages (distinct for distinct (row, tile) pairs in
 * use) before a call touches the tile, and keeps the table unchanged while
 * calls that read it run.  An entry outside [0, num_pages) for a tile a call
 * touches is not followed: the call sets status word [2], reads page 0 for the
 * attention, and skips the append's write.  Everything else (appends, decode,
 * the fused call, all modes) is the same as for the contiguous layout. */
size_t rq_cache_paged_bytes(const rq_config* cfg, int32_t num_pages);   /* 0 if invalid */

/*   dev_pool     device, >= rq_cache_paged_bytes(cfg, num_pages), 16-byte aligned
 *   block_table  device int32 [max_batch][max_tiles_per_row], 16-byte aligned,
 *                max_tiles_per_row >= ceil(max_seq_len / 64); caller-owned
 *   R_dev, out   as rq_cache_create
 * Errors: INVALID_ARG (null, num_pages <= 0, table too narrow), UNSUPPORTED,
 * CAPACITY, ALIGNMENT, CUDA. */
rq_status rq_cache_create_paged(const rq_config* cfg, int32_t num_pages, void* dev_pool, size_t bytes,
                                const int32_t* block_table, int32_t max_tiles_per_row, const float* R_dev,
                                rq_cache** out);

/* Free the host handle (not the caller's device memory).  NULL is accepted. */
rq_status rq_cache_destroy(rq_cache* cache);

/* Compress n_tokens new tokens of one (layer, group) for rows 0..batch-1 and
 * write them at positions seq_lens[b] .. seq_lens[b] + n_tokens - 1.
 * Follows the explainer's stored-overlay paragraph: anchor = last loop, INT4;
 * every earlier loop: LS coefficient (BF16), rotated residual, INT2.
 *   kv        device bf16 [P][2][batch][H][n_tokens][d] (loop, K/V, row, head, token, channel);
 *             at decode time this is the BF16 temporary buffer with n_tokens = 1.
 *   seq_lens  device int32 [batch], tokens already cached per row (not modified;
 *             the caller advances it afterwards).  Every seq_lens[b] + n_tokens
 *             must be <= max_seq_len: the host cannot see device values, so the
 *             kernel skips a row that would overflow and sets status[1] = 1.
 *   status    device int32[4] or NULL; see the status word under
 *             rq_decode_workspace_bytes (the workspace's first 16 bytes serve).
 * Errors: INVALID_ARG, CAPACITY (batch > max_batch or n_tokens > max_seq_len),
 * ALIGNMENT, UNSUPPORTED (batch * num_heads > 65535), CUDA. */
rq_status rq_append(rq_cache* cache, int32_t layer, int32_t group, int32_t batch,
                    const void* kv, const int32_t* seq_lens, int32_t n_tokens,
                    int32_t* status, void* stream);

/* Workspace (device bytes) one rq_decode_attention call needs for `batch` rows
 * on the current device.  The workspace must be zero-filled once before its
 * first use (the status word must start at zero).  Its first 16 bytes
 * are the status word (int32[4]): [0] != 0 after a device-side wait timed out,
 * [1] != 0 after an append skipped a row that would overflow, [2] != 0 after a
 * call met a block-table entry outside the page pool (paged layout). */
size_t rq_decode_workspace_bytes(const rq_config* cfg, int32_t batch);

/* One decode-attention call: query loop `loop` (0-based; loop == P-1 is the
 * anchor loop) of (layer, group), for rows 0..batch-1, all heads.
 * Keys/values are the seq_lens[b] cached tokens rebuilt for this loop, plus
 * the current token's BF16 K/V (the temporary buffer: the explainer's paragraph
 * on why the last-loop anchor forces the current token to stay in BF16).
 *   q              device bf16 [batch][H][d]
 *   k_cur, v_cur   device bf16 [batch][H][d], this loop's K/V of the current token
 *   seq_lens       device int32 [batch]
 *   softmax_scale  e.g. 1/sqrt(d)
 *   out            device float32 [batch][H][d]
 *   workspace      device, >= rq_decode_workspace_bytes(cfg, batch), zeroed once
 * Split-K over the sequence: each CTA of a balanced grid streams its range of
 * tiles into one partial softmax state per (CTA, row, head); a merge kernel
 * then combines the partial softmax
 * states, adds the current token and applies R^T once.
 * Chained mode reads the anchor and every residual plane from this loop to
 * the anchor; decode supports it for loops_per_group <= 8 (UNSUPPORTED beyond,
 * and for head_dim 128 with group_size 16 and 8 loops: one call's working set
 * would not fit one SM's shared memory).
 * Errors: INVALID_ARG, CAPACITY (batch > max_batch), WORKSPACE, ALIGNMENT,
 * UNSUPPORTED, CUDA. */
rq_status rq_decode_attention(rq_cache* cache, int32_t layer, int32_t group, int32_t loop,
                              int32_t batch, const void* q, const void* k_cur, const void* v_cur,
                              const int32_t* seq_lens, float softmax_scale, float* out,
                              void* workspace, size_t workspace_bytes, void* stream);

/* The group's last-loop (anchor-loop) call and the current token's append in
 * one call: the same output as rq_decode_attention(loop = P-1) and then the
 * same cache bytes as rq_append(n_tokens = 1) with the same kv_cur.  The
 * explainer's temporary-buffer paragraph: the current token of every loop
 * stays in BF16 until the anchor loop has produced its K/V; that is the moment
 * this call compresses it.  The merge kernel of the call does the append, one
 * CTA per (row, head); it computes while the attention kernel still streams
 * the cache and writes the new slot only after that kernel has finished.
 *   q          device bf16 [batch][H][d], query of loop P-1
 *   kv_cur     device bf16 [P][2][batch][H][d] (loop, K/V, row, head, channel):
 *              the current token of every loop (rq_append's kv with
 *              n_tokens = 1); its loop P-1 blocks are the attention's k_cur, v_cur
 *   seq_lens   device int32 [batch]: tokens already cached; the attention reads
 *              them and the token is written at position seq_lens[b] (not
 *              modified; the caller advances it afterwards).  A row with
 *              seq_lens[b] + 1 > max_seq_len is attended but not appended, and
 *              the workspace's status word gets [1] = 1.
 *   softmax_scale, out, workspace, workspace_bytes: as rq_decode_attention
 * Errors: as rq_decode_attention. */
rq_status rq_decode_attention_append(rq_cache* cache, int32_t layer, int32_t group, int32_t batch,
                                     const void* q, const void* kv_cur, const int32_t* seq_lens,
                                     float softmax_scale, float* out, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Rows one decode call (rq_decode_attention, _append, _noalloc, _bf16) may
 * cover; a larger batch returns RQ_ERR_UNSUPPORTED (split it into calls). */
#define RQ_MAX_DECODE_BATCH 256

/* Size of the workspace built into the library for rq_decode_attention_noalloc
 * (2 MiB of device memory, held on every device that loads the library until
 * the process exits).  With 152 SMs and head_dim 128 it covers batch *
 * num_query_heads up to about 740 (row, head) pairs (split-K partials of
 * 1040 B and a query pack of 1152 B per pair, plus 456 CTA partials). */
#define RQ_NOALLOC_WORKSPACE_BYTES (2u * 1024u * 1024u)

/* rq_decode_attention for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point.  Some callers are handed
 * their buffers and may not allocate more: a plugin whose host application
 * owns all device memory, a process under a memory budget fixed up front,
 * or a path on which an allocation could block or fail.  This call takes
 * the same arguments as rq_decode_attention, less the workspace, and
 * performs no device allocation: its scratch (status word, split-K
 * partials, query packs) lives in one array of RQ_NOALLOC_WORKSPACE_BYTES inside
 * the library.
 *   status   device int32[4] or NULL: receives the call's status word (as
 *            under rq_decode_workspace_bytes) on `stream` after the kernel.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any
 * stream capture.  Each call clears the part of the array it uses on
 * `stream` before its kernel, then runs the same kernel as
 * rq_decode_attention.  All calls share the one array: calls that overlap
 * on the GPU (other streams, other host threads) race and give wrong
 * results, so serialize them.  On one stream the clear is an ordinary
 * stream operation: it starts after the previous call's kernels have
 * finished, so consecutive noalloc calls do not overlap their start with
 * the previous call's tail the way rq_decode_attention calls with
 * workspaces do.  The status copied to `status` is the current call's only
 * (the clear zeroes the word first); a caller that wants to know whether
 * any of several calls failed ORs the words it receives.
 * Errors: as rq_decode_attention; WORKSPACE when the call needs more than
 * RQ_NOALLOC_WORKSPACE_BYTES (too many rows x heads for the built-in array;
 * use rq_decode_attention with a workspace of rq_decode_workspace_bytes). */
rq_status rq_decode_attention_noalloc(rq_cache* cache, int32_t layer, int32_t group,
                                      int32_t loop, int32_t batch, const void* q,
                                      const void* k_cur, const void* v_cur,
                                      const int32_t* seq_lens, float softmax_scale, float* out,
                                      int32_t* status, void* stream);

/* Workspace (device bytes) for rq_decode_attention_bf16; same zero-once rule. */
size_t rq_bf16_workspace_bytes(int32_t batch, int32_t num_heads, int32_t head_dim);

/* Uncompressed comparator: the same split-K decode attention over plain BF16
 * K/V (the role the pages give vLLM's BF16 FlashAttention baseline).
 *   k_cache, v_cache  device bf16 [batch][H][max_seq][d]
 *   k_cur, v_cur, q   device bf16 [batch][H][d]
 *   seq_lens          device int32 [batch] (each <= max_seq)
 *   out               device float32 [batch][H][d]
 * Errors: INVALID_ARG, UNSUPPORTED (head_dim), WORKSPACE, ALIGNMENT, CUDA. */
rq_status rq_decode_attention_bf16(const void* k_cache, const void* v_cache,
                                   const void* k_cur, const void* v_cur, const void* q,
                                   const int32_t* seq_lens, int32_t batch, int32_t num_heads,
                                   int32_t head_dim, int32_t max_seq, float softmax_scale,
                                   float* out, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Static description of a status code (never NULL). */
const char* rq_status_string(rq_status status);

#ifdef __cplusplus
}
#endif
#endif /* RQ_H_ */

/*
 * dsa.h — C ABI of the GB300 (sm_103a) DSA layer-step library.
 *
 * The computation (vLLM blog post "vLLM delivers day-0 support for Kimi K3.1 Pro",
 * section "Sparse Attention in K3.1 Pro" and Figure 1): a lightning indexer keeps
 * one FP8 key per token (132 bytes with its scale) and scores every earlier token
 * for each query with 32 light heads; the 2,048 best tokens are kept; MLA
 * attention with 96 absorbed query heads then runs exactly, but only over those
 * tokens' 576-byte latents.  The cache layout follows "A KV cache for three kinds
 * of state": one contiguous row per cache block holds that block's index-key page
 * and latent page at fixed offsets, and block tables are translated into page
 * addresses (here: inside the kernels).  MXFP4 index keys (68 B/token) follow
 * "AMD / Quantization: Native MXFP4 indexer"; NVFP4 latents (352 B/token) follow
 * "KV cache footprint".
 *
 * Conventions for every call:
 *  - Pointers documented "device" must point to device memory of the current
 *    CUDA device; the caller owns every buffer, including the workspace.  The
 *    library allocates no memory and keeps no state across calls (what a call
 *    leaves in the workspace is a hint at most, see dsa_layer_step).
 *  - Calls are asynchronous and ordered on `stream` (a cudaStream_t; 0 = legacy
 *    default stream).  A return value of DSA_OK means the work was validated
 *    and enqueued; device-side findings (a block id outside the pool, a wait
 *    that timed out) are recorded in the workspace's status word and reported
 *    by dsa_check().
 *  - Arguments are validated on the host before anything is enqueued; on an
 *    error nothing is enqueued.  No C++ exception crosses this interface.
 *  - Shapes: T query tokens, B requests, k = topk <= 2048, indexer 32 heads x
 *    128 dims, MLA 96 heads, latent 576 dims of which the first 512 are the value.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dsa_stream_t; /* identical to cudaStream_t */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = -1,  /* a null pointer, bad size, misaligned address or range */
  DSA_ERR_UNSUPPORTED = -2,  /* a valid but unsupported format / block size / device */
  DSA_ERR_CUDA = -3,         /* a CUDA runtime or driver call failed */
  DSA_ERR_WORKSPACE = -4,    /* workspace null, misaligned or smaller than required */
  DSA_ERR_TIMEOUT = -5,      /* a bounded device-side wait gave up (dsa_check) */
  DSA_ERR_DEVICE_CHECK = -6  /* a device-side range check failed (dsa_check) */
} dsa_status;

enum { DSA_IDX_FP8 = 0, DSA_IDX_MXFP4 = 1 };  /* index-key page formats */
enum { DSA_LAT_FP8 = 0, DSA_LAT_NVFP4 = 1 };  /* latent page formats */

#define DSA_IDX_HEADS 32
#define DSA_IDX_DIM 128
#define DSA_MLA_HEADS 96
#define DSA_LAT_DIM 576
#define DSA_V_DIM 512
#define DSA_MAX_TOPK 2048
#define DSA_ABI_VERSION 1

/*
 * One DSA layer's view of the packed KV pool.
 *
 * Row r starts at pool + r * row_stride_bytes.  For a block of `block_size`
 * tokens (a power of two, 16..256) the index page at row + idx_page_offset is
 *   FP8  : block_size x 128 e4m3 value bytes, then block_size x fp32 scales
 *          (little endian); key(s) = e4m3(code) * scale(s)          (132 B/token)
 *   MXFP4: block_size x 64 bytes of packed e2m1 (element 2i in the low nibble of
 *          byte i), then block_size x 4 E8M0 bytes (scale j covers dims 32j..32j+31)
 *                                                                   (68 B/token)
 * and the latent page at row + lat_page_offset is
 *   FP8  : block_size x 576 e4m3 bytes                              (576 B/token)
 *   NVFP4: block_size x 352-byte records: 288 bytes packed e2m1, 36 e4m3 scales
 *          (scale j covers dims 16j..16j+15), 28 bytes of padding (352 B/token)
 * Token s of request b lives in row block_table[b][s / block_size], slot
 * s % block_size.  pool, row_stride_bytes and both offsets must be multiples of
 * 16 bytes; with MXFP4 index keys pool, row_stride_bytes and idx_page_offset must
 * be multiples of 32 bytes.  Index-key scales must be finite; latents and keys must hold no NaN
 * codes.  The pool is device memory owned by the caller and only read.
 */
typedef struct {
  const void *pool;          /* device */
  int64_t num_rows;          /* rows in the pool; block ids must lie in [0, num_rows) */
  int64_t row_stride_bytes;
  int64_t idx_page_offset;
  int64_t lat_page_offset;
  int32_t block_size;
  int32_t idx_fmt;           /* DSA_IDX_* */
  int32_t lat_fmt;           /* DSA_LAT_* */
  int32_t reserved;          /* must be 0 */
} dsa_kv_layout;

/*
 * The query batch.  Query token t belongs to request q_req[t] and sits at
 * absolute position q_pos[t] of that request; it attends to positions
 * 0..q_pos[t] (causal and inclusive: the new tokens' keys and latents are in the
 * cache before the call).  Requirements (checked on the device; a violation sets
 * DSA_ERR_DEVICE_CHECK): 0 <= q_req[t] < num_reqs, 0 <= q_pos[t] < ctx_lens[q_req[t]]
 * <= max_ctx_len <= bt_stride * block_size.  All pointers are device memory.
 * Tokens of one request should be contiguous in t so the indexer can share key
 * reads across them; any order is correct.
 *
 * Batch invariance ("Zero-mismatch RL on day 0": a token's result must not
 * depend on its batch).  The indexer scores and the top-k selection of a token
 * never depend on the rest of the batch.  The attention output is split over
 * the selected list into a number of partials chosen from the batch size (to
 * fill the GPU); with DSA_BATCH_INVARIANT set the split is fixed (one partial
 * per 128 selected tokens) so the output is bit-identical for any batch, at the
 * cost of more partial traffic for large batches.
 */
#define DSA_BATCH_INVARIANT 1
/*
 * MXFP4 index queries ("Low-latency decode: a fused DSA decode path": the index
 * query is quantized to FP8 or MXFP4).  With this flag q_idx of every call that
 * takes it holds T x 32 x 64 bytes of packed e2m1 codes (head h of token t at
 * (t * 32 + h) * 64, element 2i in the low nibble of byte i), then T x 32 x 4 E8M0
 * exponents (byte j of head h of token t at T * 2048 + (t * 32 + h) * 4 + j covers
 * dims 32j..32j+31): 68 bytes per head, 32-byte aligned.  The query value is
 * e2m1(code) * 2^(E - 127); the head weights are used as given.  Only with MXFP4
 * index keys (DSA_ERR_UNSUPPORTED otherwise); dsa_indexer_front then writes this
 * form.  Without the flag q_idx holds e4m3 codes [T, 32, 128].
 */
#define DSA_BATCH_QIDX_MXFP4 2
typedef struct {
  int32_t num_tokens;        /* T >= 0 */
  int32_t num_reqs;          /* B >= 1 */
  const int32_t *q_req;      /* [T] */
  const int32_t *q_pos;      /* [T] */
  const int32_t *ctx_lens;   /* [B] */
  const int32_t *block_table;/* [B, bt_stride] row ids */
  int32_t bt_stride;
  int32_t flags;             /* DSA_BATCH_* bits; 0 = default */
  int64_t max_ctx_len;       /* host-side upper bound of ctx_lens, used for sizing */
} dsa_batch;

/* ABI version of the loaded library (DSA_ABI_VERSION). */
int32_t dsa_abi_version(void);

/* Human-readable name of a status code (static storage). */
const char *dsa_status_string(dsa_status status);

/*
 * The CUDA error behind the last DSA_ERR_CUDA that a call returned on the
 * calling host thread: the cudaError_t value of the failing runtime call (0 if
 * none yet), or -1 when encoding a TMA tensor map failed.  If `name` is not
 * NULL it receives the error's name (static storage).  Later successful calls
 * do not clear it.
 */
int32_t dsa_last_cuda_error(const char **name);

/*
 * Bytes of device workspace the calls below need for this layout/batch/topk
 * (the maximum over all calls; 256-byte aligned).  0 on invalid arguments.
 * The first 256 bytes hold the status word, which persists across calls until
 * dsa_check() clears it: zero the workspace once after allocating it.
 */
size_t dsa_workspace_size(const dsa_kv_layout *layout, const dsa_batch *batch, int32_t topk);

/*
 * Indexer scores ("Sparse Attention in K3.1 Pro"):
 *   scores[t * ld_scores + s] = sum_{h<32} w[t,h] * ReLU(q_idx[t,h,:] . key(s)),
 * for s = 0..q_pos[t], with key(s) the dequantised index key of token s of
 * request q_req[t].  Entries beyond q_pos[t] are not written.
 *  q_idx : device, e4m3 codes [T, 32, 128] (16-byte aligned); used as-is (any
 *          query-side scale belongs in w)
 *  w     : device, fp32 [T, 32]
 *  scores: device, fp32 [T, ld_scores], ld_scores >= max_ctx_len, 16-byte aligned rows
 * Keys are scored with FP8 tensor-core MMAs (fp32 accumulation); the key scale
 * is applied after the head reduction (exact for a positive or negative scale).
 */
dsa_status dsa_indexer_score(const dsa_kv_layout *layout, const dsa_batch *batch,
                             const void *q_idx, const float *w, float *scores,
                             int64_t ld_scores, void *workspace, size_t workspace_bytes,
                             dsa_stream_t stream);

/*
 * Exact top-k ("Sparse Attention in K3.1 Pro": the best 2,048 tokens are kept): for each token t, the k
 * largest of scores[t, 0..q_pos[t]]; equal scores are ordered by lower position
 * first (-0.0 equals +0.0).  idx[t, :] receives the selected positions in
 * ascending order; when q_pos[t] + 1 < k every position is selected and the
 * tail is filled with -1.  The result is deterministic and independent of the
 * rest of the batch.
 *  scores    : device fp32 [T, ld_scores] (not modified); NaN scores are unsupported
 *  idx       : device int32 [T, topk]
 *  phys_slots: device int32 [T, topk] or NULL: for each selected position s the
 *              physical cache slot block_table[b][s/bs] * bs + s % bs (-1 for padding);
 *              needs `layout` (only its block_size is read); `layout` may be NULL
 *              when phys_slots is NULL.
 */
dsa_status dsa_topk(const dsa_kv_layout *layout, const dsa_batch *batch, const float *scores,
                    int64_t ld_scores, int32_t topk, int32_t *idx, int32_t *phys_slots,
                    void *workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * Sparse MLA ("Sparse Attention in K3.1 Pro": exact attention restricted to the kept tokens):
 * for each token t and head h < 96, over the positions S_t = {idx[t, i] >= 0}:
 *   logit(s) = sm_scale * q[t,h,:] . c(s)          (all 576 dims)
 *   out[t,h,:] = sum_s softmax(logit)(s) * c(s)[0:512]
 *   lse[t,h]  = ln sum_s exp(logit(s))
 * with c(s) the dequantised latent of position s of request q_req[t].
 *  q  : device bf16 [T, 96, 576] (16-byte aligned)
 *  idx: device int32 [T, topk]; valid entries first, then -1 (as dsa_topk writes
 *       them); every valid entry must be <= q_pos[t]; at least one per token
 *  out: device bf16 [T, 96, 512];  lse: device fp32 [T, 96] or NULL
 * QK runs as bf16 x bf16 (the e4m3 latent is exact in bf16) and PV as fp16 P x
 * fp16 V on the tensor cores with fp32 accumulation; per-split partials are
 * merged by log-sum-exp in fp32.
 */
dsa_status dsa_sparse_mla(const dsa_kv_layout *layout, const dsa_batch *batch, const void *q,
                          const int32_t *idx, int32_t topk, float sm_scale, void *out,
                          float *lse, void *workspace, size_t workspace_bytes,
                          dsa_stream_t stream);

/*
 * The whole DSA layer step: indexer scores -> exact top-k -> sparse MLA, with
 * the intermediate scores and indices kept in the workspace.
 *  idx_out: device int32 [T, topk] or NULL — receives the selected positions
 *  other arguments as in the three calls above.
 * The scorer also counts each token's scores by their top 11 key bits into the
 * workspace, and the top-k starts its radix select from those counts and leaves
 * them zeroed for the next step.  The counts are checked exactly before use:
 * whatever the workspace held beforehand, the results are the same (a workspace
 * that was not left zeroed only costs the top-k an extra pass).
 */
dsa_status dsa_layer_step(const dsa_kv_layout *layout, const dsa_batch *batch,
                          const void *q_idx, const float *w, const void *q, int32_t topk,
                          float sm_scale, int32_t *idx_out, void *out, float *lse,
                          void *workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * The layer step for a caller whose per-step inputs and outputs live in host
 * memory.  The vLLM post ("Sparse Attention in K3.1 Pro") defines only the
 * device-side step; this call adds the transfers around it.  All of it is
 * ordered on `stream`:
 *  1. the host inputs are copied into the device buffers that the other arguments
 *     and `batch` name (q_req, q_pos, ctx_lens and block_table are overwritten on
 *     the device);
 *  2. dsa_layer_step runs, with the same arguments and results;
 *  3. out, and lse and idx where `host` asks for them, are copied back.
 * Each array is copied on its own, unless host->flags holds DSA_HOST_PACKED.  With
 * that flag, the caller promises that the inputs q, q_idx, w, q_req, q_pos,
 * ctx_lens and block_table lie back to back in this order, in one host allocation
 * and in one device allocation.  They then move as a single copy.  The call checks
 * that each array starts where the one before it ends, on both sides, and returns
 * DSA_ERR_INVALID_ARG where one does not.  Whether the arrays share an allocation
 * cannot be checked: a copy must not span two allocations.  Host memory should be
 * page-locked: a range that lies inside one page-locked allocation the device can
 * address (cudaHostAlloc, cudaMallocHost, cudaHostRegister; checked with the
 * driver's pointer attributes) is moved by the library's copy kernel through its
 * mapped device address, all such inputs in one launch and all such outputs in
 * another.  Any other host memory goes through cudaMemcpyAsync: the results are
 * the same, but with pageable memory the host waits for each copy.
 * The call returns once everything is enqueued.  The host outputs hold the results
 * only once the stream has passed them (cudaStreamSynchronize or an event).  Every
 * argument is validated before anything is enqueued.
 *  host: host pointers, each sized like its device counterpart.  ctx_lens and
 *        block_table are always required.  q_idx, w, q, q_req, q_pos and out are
 *        required when T > 0.  lse may be NULL, and is allowed only when the
 *        device lse is given.  idx may be NULL, and is allowed only when idx_out
 *        is given.  flags: 0 or DSA_HOST_PACKED.
 */
#define DSA_HOST_PACKED 1
typedef struct {
  const void *q_idx;          /* e4m3 [T, 32, 128] */
  const float *w;             /* fp32 [T, 32] */
  const void *q;              /* bf16 [T, 96, 576] */
  const int32_t *q_req;       /* [T] */
  const int32_t *q_pos;       /* [T] */
  const int32_t *ctx_lens;    /* [B] */
  const int32_t *block_table; /* [B, bt_stride] */
  void *out;                  /* bf16 [T, 96, 512], written */
  float *lse;                 /* fp32 [T, 96] or NULL, written */
  int32_t *idx;               /* int32 [T, topk] or NULL, written */
  int32_t flags;              /* DSA_HOST_* bits */
} dsa_host_io;
dsa_status dsa_layer_step_host(const dsa_kv_layout *layout, const dsa_batch *batch, void *q_idx, float *w,
                               void *q, int32_t topk, float sm_scale, int32_t *idx_out, void *out,
                               float *lse, const dsa_host_io *host, void *workspace,
                               size_t workspace_bytes, dsa_stream_t stream);

/*
 * dsa_topk without a workspace, for callers that cannot allocate device memory
 * (code running in a stream callback or host-function node, plugins whose host
 * framework owns all allocations, loops that forbid allocator use after start-up).
 * The vLLM post describes no such call; it exists only for those callers.
 *
 * Same arguments, checks, results and guarantees as dsa_topk, minus the
 * workspace.  Rows of at most 65,536 scores (max_ctx_len <= 65,536) need no
 * scratch at all.  Longer rows need at most T x (40,988 + 8 x ceil(max_ctx_len /
 * 4096)) + 1,280 bytes for histograms, candidate lists and per-chunk counts, which
 * live in a fixed DSA_NOALLOC_SCRATCH_BYTES array of device memory inside the
 * library; every GPU that loads the library holds that array until the process
 * exits.  A batch with longer rows that needs more returns DSA_ERR_WORKSPACE
 * (up to 97 query tokens fit at 1M-token contexts, 101 just above 65,536).  The
 * call allocates nothing.
 *  - The first call in each CUDA context looks up the array's device address
 *    (cudaGetSymbolAddress with that context current); make that first call
 *    before any stream capture.  A context created later (another device, or the
 *    primary context re-created after cudaDeviceReset) gets its own lookup.
 *  - Every call uses the same array: the call clears the part that must start at
 *    zero on `stream`, but calls that overlap on the GPU (other streams, other
 *    host threads) race on it; issue them in order on one stream.
 *  - Device-side range findings are not reported (there is no workspace status
 *    word); out-of-range positions are clamped so nothing is read out of bounds.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (4u << 20)
dsa_status dsa_topk_noalloc(const dsa_kv_layout *layout, const dsa_batch *batch, const float *scores,
                            int64_t ld_scores, int32_t topk, int32_t *idx, int32_t *phys_slots,
                            dsa_stream_t stream);

/*
 * The fused indexer front ("Low-latency decode: a fused DSA decode path": one
 * kernel normalises the query, projects the indexer query, quantizes it with the
 * scales absorbed by the head weights and writes the new token's index key).  The post
 * prints no shapes; this call takes them as stated here.  For each query token t:
 *   y = c_q[t] / sqrt(mean(c_q[t]^2) + eps) * norm_weight          (RMSNorm, fp32)
 *   q[h, :] = w_qi[h * 128 .. h * 128 + 127, :] . y   (fp32 sums; y enters as bf16 hi + lo terms)
 *   s[h] = max|q[h, :]| / 448 (1 for an all-zero head)
 *   q_idx[t, h, :] = e4m3(q[h, :] / s[h]),  w_out[t, h] = head_w[t, h] * s[h]
 * so q_idx and w_out are the inputs dsa_indexer_score / dsa_layer_step take.
 * With DSA_BATCH_QIDX_MXFP4 (MXFP4 index pages only) q_idx is written in that
 * flag's layout instead: per head and 32-dim block b, E = floor(log2 max|q|) - 2
 * + 127 clamped to 0..254 (0 for a zero block), codes e2m1(q * 2^(127 - E))
 * (round to nearest even, saturating at 6); w_out[t, h] = head_w[t, h].
 * With k_new given, the new token's index key is written into the pool at the
 * token's own position (block_table[q_req[t]][q_pos[t] / bs], slot q_pos[t] % bs).
 * FP8 pages: s_k = max|k| / 448 in fp32 (1 when zero), 128 codes e4m3(k / s_k),
 * then s_k in the page's scale area.  MXFP4 pages: per 32 dims the exponent and
 * e2m1 codes by the rule above, 64 code bytes at the slot, 4 exponents in the
 * scale area.
 *  c_q        : device bf16 [T, d_q], d_q a multiple of 8 in 64..4096
 *  norm_weight: device bf16 [d_q];  eps >= 0
 *  w_qi       : device bf16 [32 * 128, d_q] (row h * 128 + d is output dim d of head h)
 *  head_w     : device fp32 [T, 32];  k_new: device bf16 [T, 128] or NULL
 *  q_idx      : device e4m3 [T, 32, 128], or MXFP4 (68 bytes per head, 32-byte
 *               aligned) with DSA_BATCH_QIDX_MXFP4 (written);  w_out: device fp32 [T, 32] (written)
 *  workspace  : only its status word is used (>= 256 bytes); a block id or
 *               position out of range is recorded there and nothing is written for it.
 * Unlike the other calls this one writes the pool (the new tokens' slots only).
 * All pointers 16-byte aligned.
 */
dsa_status dsa_indexer_front(const dsa_kv_layout *layout, const dsa_batch *batch, const void *c_q, int32_t d_q,
                             const void *norm_weight, float eps, const void *w_qi, const float *head_w,
                             const void *k_new, void *q_idx, float *w_out, void *workspace, size_t workspace_bytes,
                             dsa_stream_t stream);

/*
 * The new tokens' latents into the cache ("Low-latency decode: a fused DSA decode
 * path": the MLA query kernel writes the new token's latent into the KV cache;
 * "KV cache footprint": 576-byte FP8 or 352-byte NVFP4 latents).  For each query
 * token t the record at its own position (as in dsa_indexer_front) becomes
 *   FP8  : e4m3(latent[t, :]) (576 bytes, no scale)
 *   NVFP4: per 16 values j: scale_j = e4m3(max|x| / 6), codes e2m1(x / scale_j)
 *          (zero for a zero scale), packed two per byte (element 2i in the low
 *          nibble), 36 scale bytes, 28 zero bytes (352 bytes)
 * with round-to-nearest-even, saturating conversions in fp32.
 *  latent   : device bf16 [T, 576], 16-byte aligned
 *  workspace: only its status word is used (>= 256 bytes), as above.
 */
dsa_status dsa_write_latent(const dsa_kv_layout *layout, const dsa_batch *batch, const void *latent,
                            void *workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * Synchronises `stream`, reads the workspace status word written by earlier
 * calls, clears it, and returns DSA_OK, DSA_ERR_TIMEOUT or DSA_ERR_DEVICE_CHECK.
 */
dsa_status dsa_check(void *workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * Diagnostic of the failure path.  Every wait inside the library's kernels is
 * bounded: past its limit it gives up, records DSA_ERR_TIMEOUT in the workspace
 * status word, and the kernel drains what it has in flight and returns instead of
 * hanging.  A healthy step never reaches that limit (about 2 s), so this call runs
 * the same bounded wait on a barrier that nothing completes, with a limit of
 * `limit_cycles` SM clock cycles (1,000 .. 4e9).  Once the stream has passed it,
 * dsa_check() returns DSA_ERR_TIMEOUT (and the device stays usable).  The vLLM
 * post describes no such call; it exists to test the failure path.
 *  workspace: device, >= 256 bytes, 256-byte aligned (only the status word is used)
 */
dsa_status dsa_selftest_wait_timeout(void *workspace, size_t workspace_bytes, int64_t limit_cycles,
                                     dsa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_GB300_H */

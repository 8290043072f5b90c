// capi.cu — the extern "C" entry points declared in include/dsa.h: host-side
// validation, workspace carving, TMA descriptor encoding and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/dsa.h"

#include "hostcopy.cuh"
#include "mla_q.cuh"
#include "params.cuh"

using namespace dsa;

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Ws {
  size_t status = 0;
  size_t row_hist = 0;
  size_t plan_hdr = 0, groups = 0;
  size_t topk = 0;
  size_t scores = 0;
  int64_t ld = 0;
  size_t idx = 0, phys = 0;
  size_t part_o = 0, part_ml = 0;
  int nsplit = 1, tps = 16;
  bool fp8_mla = false;   // FP8 latents may take the one-tile-per-CTA FP8 kernel
  size_t m8_q = 0;        // its query terms (mla_q.cuh), [T] x 110,976 B
  int topk_nchunks = 1;
  size_t total = 0;
};

// SM count of the current device, for grid and split sizing (looked up once per
// device).  Any value gives correct results.  The default attention split follows
// it, and with it the rounding of the split combine; DSA_BATCH_INVARIANT fixes the
// split.  When no device answers (workspace sizing on a host without one) it is
// 152, a GB300's count.
int num_sms() {
  constexpr int kMaxDev = 64;
  static int cache[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
    cache[dev] = v;
  }
  return cache[dev];
}

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

dsa_status check_layout(const dsa_kv_layout* l, bool need_pool = true) {
  if (!l) return DSA_ERR_INVALID_ARG;
  if (need_pool && !l->pool) return DSA_ERR_INVALID_ARG;
  if (l->reserved != 0 || l->num_rows <= 0 || l->num_rows > (int64_t(1) << 31) - 1) return DSA_ERR_INVALID_ARG;
  if (!is_pow2(l->block_size) || l->block_size < 16 || l->block_size > 256) return DSA_ERR_UNSUPPORTED;
  if (l->idx_fmt != DSA_IDX_FP8 && l->idx_fmt != DSA_IDX_MXFP4) return DSA_ERR_INVALID_ARG;
  if (l->lat_fmt != DSA_LAT_FP8 && l->lat_fmt != DSA_LAT_NVFP4) return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(l->pool) & 15) || (l->row_stride_bytes & 15) || (l->idx_page_offset & 15) ||
      (l->lat_page_offset & 15))
    return DSA_ERR_INVALID_ARG;
  // MXFP4 index pages are read by a packed 4-bit tensor copy: 32-byte alignment
  if (l->idx_fmt == DSA_IDX_MXFP4 &&
      ((reinterpret_cast<uintptr_t>(l->pool) & 31) || (l->row_stride_bytes & 31) || (l->idx_page_offset & 31)))
    return DSA_ERR_INVALID_ARG;
  const int64_t idx_pb = int64_t(l->block_size) * (l->idx_fmt == DSA_IDX_FP8 ? 132 : 68);
  const int64_t lat_pb = int64_t(l->block_size) * (l->lat_fmt == DSA_LAT_FP8 ? 576 : 352);
  if (l->idx_page_offset < 0 || l->lat_page_offset < 0 || l->idx_page_offset + idx_pb > l->row_stride_bytes ||
      l->lat_page_offset + lat_pb > l->row_stride_bytes)
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// Bytes of q_idx for a batch: e4m3 codes, or MXFP4 codes and exponents.
size_t q_idx_bytes(const dsa_batch* b) {
  return size_t(b->num_tokens) * kIdxHeads * ((b->flags & DSA_BATCH_QIDX_MXFP4) ? kIdxDim / 2 + 4 : kIdxDim);
}

// MXFP4 queries need MXFP4 keys and a 32-byte aligned q_idx (a packed 4-bit tensor copy).
dsa_status check_qidx(const dsa_kv_layout* l, const dsa_batch* b, const void* q_idx) {
  if (!(b->flags & DSA_BATCH_QIDX_MXFP4)) return DSA_OK;
  if (l->idx_fmt != DSA_IDX_MXFP4) return DSA_ERR_UNSUPPORTED;
  if (b->num_tokens > 0 && (reinterpret_cast<uintptr_t>(q_idx) & 31)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status check_batch(const dsa_batch* b, int block_size) {
  if (!b) return DSA_ERR_INVALID_ARG;
  if (b->num_tokens < 0 || b->num_reqs < 1 || (b->flags & ~(DSA_BATCH_INVARIANT | DSA_BATCH_QIDX_MXFP4)) ||
      b->bt_stride < 1)
    return DSA_ERR_INVALID_ARG;
  if (b->num_tokens > 0 && (!b->q_req || !b->q_pos)) return DSA_ERR_INVALID_ARG;
  if (!b->ctx_lens || !b->block_table) return DSA_ERR_INVALID_ARG;
  if (b->max_ctx_len < 1 || b->max_ctx_len > (int64_t(1) << 30)) return DSA_ERR_INVALID_ARG;
  if (block_size > 0 && b->max_ctx_len > int64_t(b->bt_stride) * block_size) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

Ws plan_ws(const dsa_kv_layout* l, const dsa_batch* b, int topk) {
  Ws w;
  const int64_t T = b->num_tokens;
  size_t off = 0;
  w.status = off;
  off += kStatusBytes;
  // top-digit histograms from the scorer to the top-k of a layer step; the top-k
  // leaves them zeroed (a zeroed workspace starts them right; they are verified)
  w.row_hist = off;
  off = align_up(off + size_t(T > 0 ? T : 1) * 2048 * 4);
  w.plan_hdr = off;
  off = align_up(off + sizeof(PlanHeader));
  w.groups = off;
  off = align_up(off + size_t(T > 0 ? T : 1) * sizeof(ScoreGroup));
  w.topk_nchunks = static_cast<int>(cdiv(b->max_ctx_len, kTopkChunk));
  w.topk = off;
  off = align_up(off + topk_scratch_layout(T, w.topk_nchunks).total);
  w.ld = (b->max_ctx_len + 3) / 4 * 4;
  w.scores = off;
  off = align_up(off + size_t(T) * size_t(w.ld) * 4);
  w.idx = off;
  off = align_up(off + size_t(T) * size_t(topk > 0 ? topk : 1) * 4);
  w.phys = off;
  off = align_up(off + size_t(T) * size_t(topk > 0 ? topk : 1) * 4);
  // MLA split: enough CTAs to cover the GPU about twice
  const int ntiles = static_cast<int>(cdiv(topk > 0 ? topk : 1, kSelTile));
  int nsplit = 1;
  if (b->flags & DSA_BATCH_INVARIANT)
    nsplit = ntiles;   // fixed split: independent of the batch
  else if (T > 0)
    nsplit = static_cast<int>(cdiv(2 * num_sms(), T));
  if (nsplit > ntiles) nsplit = ntiles;
  if (nsplit < 1) nsplit = 1;
  w.tps = static_cast<int>(cdiv(ntiles, nsplit));
  w.nsplit = static_cast<int>(cdiv(ntiles, w.tps));
  // The FP8 kernel gives every 128 selected tokens their own CTA; it is used
  // when that fills the GPU at most about twice, and always with
  // DSA_BATCH_INVARIANT (its split never depends on the batch).
  w.fp8_mla = l->lat_fmt == DSA_LAT_FP8 &&
              ((b->flags & DSA_BATCH_INVARIANT) || T * int64_t(ntiles) <= 2 * int64_t(num_sms()));
  w.m8_q = off;
  if (w.fp8_mla) {
    off = align_up(off + size_t(T) * kQTokenBytes);
  }
  // split partials: the FP8 kernel writes one per tile
  const int part_splits = w.fp8_mla && ntiles > w.nsplit ? ntiles : w.nsplit;
  w.part_o = off;
  if (part_splits > 1) off = align_up(off + size_t(T) * part_splits * kMlaHeads * kVDim * 2);
  w.part_ml = off;
  if (part_splits > 1) off = align_up(off + size_t(T) * part_splits * kMlaHeads * 8);
  w.total = off;
  return w;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over the index-key values of every page: {128 dims, block slots, rows},
// 128-byte swizzle, 128 B per key in shared memory, ready for the MMA.  FP8 keys
// are 128 e4m3 bytes.  MXFP4 keys (64 bytes of packed e2m1 in the page) use the
// 16 x 4-bit element type that pads every 8 bytes of codes to 16 (the MMA's E2M1
// operand layout); it needs the page and the row stride 32-byte aligned, and a
// copy counts the 64 packed bytes per key.
bool make_key_map(CUtensorMap* m, const dsa_kv_layout* l) {
  auto enc = encode_fn();
  if (!enc) return false;
  const bool mx = l->idx_fmt == DSA_IDX_MXFP4;
  const int box_rows = l->block_size < kKeyTile ? l->block_size : kKeyTile;
  cuuint64_t dims[3] = {128, cuuint64_t(l->block_size), cuuint64_t(l->num_rows)};
  cuuint64_t strides[2] = {cuuint64_t(mx ? 64 : 128), cuuint64_t(l->row_stride_bytes)};
  cuuint32_t box[3] = {128, cuuint32_t(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  void* base = const_cast<uint8_t*>(static_cast<const uint8_t*>(l->pool)) + l->idx_page_offset;
  return enc(m, mx ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q_idx [T*32 rows of 128 dims], box = one token's 32 heads, 128 B per head in shared
// memory (128-byte swizzle): e4m3 codes, or MXFP4 codes (64 packed bytes per head)
// through the 16 x 4-bit element type that pads each 8 bytes of codes to 16.
bool make_qidx_map(CUtensorMap* m, const void* q_idx, int T, bool mx) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, cuuint64_t(T) * kIdxHeads};
  cuuint64_t strides[1] = {cuuint64_t(mx ? 64 : 128)};
  cuuint32_t box[2] = {128, kIdxHeads};
  cuuint32_t es[2] = {1, 1};
  return enc(m, mx ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<void*>(q_idx), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [T*96 rows, 576 bf16], box = 64 dims x 96 heads.
bool make_q_map(CUtensorMap* m, const void* q, int T) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {kLatDim, cuuint64_t(T) * kMlaHeads};
  cuuint64_t strides[1] = {kLatDim * 2};
  cuuint32_t box[2] = {64, kMlaHeads};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The FP8 attention's split partials [rows = T * nsplit * 512 dims][96 heads] fp16,
// box 32 heads x 256 rows, 64-byte swizzle (tensor stores from shared memory).
bool make_part_map(CUtensorMap* m, void* part_o, int64_t rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cuuint64_t(kMlaHeads), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(kMlaHeads) * 2};
  cuuint32_t box[2] = {32, 256};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, part_o, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// The split partials as [T * nsplit][512 dims][96 heads] fp16 for the combine: a box
// is four consecutive splits of 32 dims x 96 heads (no swizzle, 192-byte rows).
bool make_comb_map(CUtensorMap* m, void* part_o, int64_t T, int nsplit) {
  constexpr cuuint32_t kBoxSplits = 4;   // the combine's splits per copy
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(kMlaHeads), cuuint64_t(kVDim), cuuint64_t(T) * cuuint64_t(nsplit)};
  cuuint64_t strides[2] = {cuuint64_t(kMlaHeads) * 2, cuuint64_t(kMlaHeads) * 2 * kVDim};
  cuuint32_t box[3] = {cuuint32_t(kMlaHeads), 32, kBoxSplits};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, part_o, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// The indexer query projection W [4096 rows, d_q] bf16 for the front: a box is 64
// dims (128 bytes) of one head's 128 rows, 128-byte swizzle (the MMA's A operand,
// K-major); dims past d_q read as zeros.
bool make_front_w_map(CUtensorMap* m, const void* w, int d_q) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cuuint64_t(d_q), cuuint64_t(kIdxHeads) * kIdxDim};
  cuuint64_t strides[1] = {cuuint64_t(d_q) * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

PoolView pool_view(const dsa_kv_layout* l) {
  PoolView v;
  v.pool = static_cast<const uint8_t*>(l->pool);
  v.num_rows = l->num_rows;
  v.row_stride = l->row_stride_bytes;
  v.idx_off = l->idx_page_offset;
  v.lat_off = l->lat_page_offset;
  v.bs = l->block_size;
  int lg = 0;
  while ((1 << lg) < l->block_size) ++lg;
  v.log2_bs = lg;
  v.idx_fmt = l->idx_fmt;
  v.lat_fmt = l->lat_fmt;
  return v;
}

BatchView batch_view(const dsa_batch* b) {
  BatchView v;
  v.T = b->num_tokens;
  v.B = b->num_reqs;
  v.q_req = b->q_req;
  v.q_pos = b->q_pos;
  v.ctx_lens = b->ctx_lens;
  v.bt = b->block_table;
  v.bt_stride = b->bt_stride;
  v.max_ctx = static_cast<int32_t>(b->max_ctx_len);
  return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

dsa_status check_ws(void* ws, size_t bytes, const Ws& w) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return DSA_ERR_WORKSPACE;
  if (bytes < w.total) return DSA_ERR_WORKSPACE;
  return DSA_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// The CUDA error behind the last DSA_ERR_CUDA returned on this host thread.
thread_local int32_t g_last_cuda = 0;
thread_local const char* g_last_cuda_name = "no error";

dsa_status cuda_fail(cudaError_t e) {
  g_last_cuda = static_cast<int32_t>(e);
  g_last_cuda_name = cudaGetErrorName(e);
  return DSA_ERR_CUDA;
}

dsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : cuda_fail(e); }

dsa_status encode_fail() {
  g_last_cuda = -1;
  g_last_cuda_name = "TMA descriptor encoding failed";
  return DSA_ERR_CUDA;
}

// `row_hist`: the top-k hint histograms to add to, or null.
// `mla_q`: the layer step's absorbed query when its attention runs on FP8 latents
// (the scorer then also writes the attention's query terms), else null.
dsa_status run_indexer(const dsa_kv_layout* l, const dsa_batch* b, const void* q_idx, const float* w, float* scores,
                       int64_t ld, void* ws, const Ws& wl, cudaStream_t st, uint32_t* row_hist = nullptr,
                       const void* mla_q = nullptr) {
  const int T = b->num_tokens;
  if (T == 0) return DSA_OK;
  const bool qmx = (b->flags & DSA_BATCH_QIDX_MXFP4) != 0;
  CUtensorMap kmap, qmap;
  if (!make_key_map(&kmap, l) || !make_qidx_map(&qmap, q_idx, T, qmx)) return encode_fail();
  const int G = indexer_group_size(l->idx_fmt, T == b->num_reqs);
  const bool direct = G == 1 && T <= kDirectMaxT;
  uint32_t* status = at<uint32_t>(ws, wl.status);
  BatchView bv = batch_view(b);
  if (!direct) {
    cudaError_t e = cudaMemsetAsync(at<uint8_t>(ws, wl.plan_hdr), 0,
                                    wl.groups + size_t(T) * sizeof(ScoreGroup) - wl.plan_hdr, st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_plan_groups(bv, G, at<ScoreGroup>(ws, wl.groups), at<PlanHeader>(ws, wl.plan_hdr), status, st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  IndexerParams p;
  p.pool = pool_view(l);
  p.b = bv;
  p.w = w;
  p.scores = scores;
  p.ld = ld;
  p.hdr = at<PlanHeader>(ws, wl.plan_hdr);
  p.groups = at<ScoreGroup>(ws, wl.groups);
  p.status = status;
  p.direct = direct ? 1 : 0;
  p.row_hist = G == 1 ? row_hist : nullptr;
  p.mla_q = static_cast<const __nv_bfloat16*>(mla_q);
  p.mla_q_terms = mla_q ? at<uint8_t>(ws, wl.m8_q) : nullptr;
  p.qmx = qmx ? 1 : 0;
  p.q_scales = qmx ? static_cast<const uint8_t*>(q_idx) + size_t(T) * kIdxHeads * (kIdxDim / 2) : nullptr;
  return cuda_status(launch_indexer(kmap, qmap, p, G, num_sms(), st));
}

// `chained`: the launch follows a kernel of this library on the stream (see launch_ex).
// `pre_hist`: histograms the scorer left for these scores, or null.
dsa_status run_topk(const dsa_kv_layout* l, const dsa_batch* b, const float* scores, int64_t ld, int topk,
                    int32_t* idx, int32_t* phys, void* ws, const Ws& wl, cudaStream_t st, bool chained,
                    uint32_t* pre_hist = nullptr, bool zeroed = false) {
  if (b->num_tokens == 0) return DSA_OK;
  TopkParams p;
  p.b = batch_view(b);
  p.scores = scores;
  p.ld = ld;
  p.k = topk;
  topk_bind_scratch(p, at<uint8_t>(ws, wl.topk), topk_scratch_layout(b->num_tokens, wl.topk_nchunks),
                    wl.topk_nchunks);
  p.idx = idx;
  p.phys = phys;
  int lg = 0;
  if (l)
    while ((1 << lg) < l->block_size) ++lg;
  p.log2_bs = lg;
  p.status = at<uint32_t>(ws, wl.status);
  p.pre_hist = pre_hist;
  return cuda_status(launch_topk(p, st, chained, zeroed));
}

// Whether the attention of this plan takes the FP8 kernel on this device.
bool use_fp8_mla(const Ws& wl) { return wl.fp8_mla && sparse_mla_fp8_available(); }

// `in_step`: inside a layer step, whose scorer has written the FP8 kernel's query
// terms; otherwise a small kernel writes them first.
dsa_status run_mla(const dsa_kv_layout* l, const dsa_batch* b, const void* q, const int32_t* idx,
                   const int32_t* phys, int topk, float sm_scale, void* out, float* lse, void* ws, const Ws& wl,
                   cudaStream_t st, bool chained, bool in_step = false) {
  const int T = b->num_tokens;
  if (T == 0) return DSA_OK;
  MlaParams p;
  p.pool = pool_view(l);
  p.b = batch_view(b);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.idx = idx;
  p.phys = phys;
  p.topk = topk;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.tps = wl.tps;
  p.nsplit = wl.nsplit;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.part_o = at<__half>(ws, wl.part_o);
  p.part_ml = at<float2>(ws, wl.part_ml);
  p.status = at<uint32_t>(ws, wl.status);
  if (use_fp8_mla(wl)) {
    p.nsplit = static_cast<int>(cdiv(topk, kSelTile));   // one tile per CTA (the plan sized the partials so)
    p.tps = 1;
    p.q_terms = at<uint8_t>(ws, wl.m8_q);
    if (!in_step) {
      const cudaError_t e = launch_mla_qprep(p.q, at<uint8_t>(ws, wl.m8_q), T, st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    CUtensorMap pmap, cmap;
    std::memset(&pmap, 0, sizeof(pmap));
    std::memset(&cmap, 0, sizeof(cmap));
    if (p.nsplit > 1 && (!make_part_map(&pmap, p.part_o, int64_t(T) * p.nsplit * kVDim) ||
                         !make_comb_map(&cmap, p.part_o, T, p.nsplit)))
      return encode_fail();
    return cuda_status(launch_sparse_mla_fp8(pmap, cmap, p, st, chained));
  }
  CUtensorMap qmap, cmap;
  std::memset(&cmap, 0, sizeof(cmap));
  if (!make_q_map(&qmap, q, T)) return encode_fail();
  if (p.nsplit > 1 && !make_comb_map(&cmap, p.part_o, T, p.nsplit)) return encode_fail();
  return cuda_status(launch_sparse_mla(qmap, cmap, p, st, chained));
}

// The device address of the host range [host, host + bytes) when the whole range
// lies inside one page-locked allocation that the current device can address
// (cudaHostAlloc, cudaMallocHost or cudaHostRegister), else null: only such a
// range is handed to the copy kernel; anything else goes through cudaMemcpyAsync.
void* mapped_device_ptr(const void* host, size_t bytes) {
  using Fn = CUresult (*)(void*, CUpointer_attribute, CUdeviceptr);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(f);
  });
  if (!fn || !host || !bytes) return nullptr;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    (void)cudaGetLastError();   // not a pointer the runtime knows: no error left behind
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  const CUdeviceptr d = reinterpret_cast<CUdeviceptr>(a.devicePointer);
  CUdeviceptr start = 0;
  size_t size = 0;
  if (fn(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, d) != CUDA_SUCCESS ||
      fn(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, d) != CUDA_SUCCESS)
    return nullptr;
  if (d < start || d - start > size || bytes > size - (d - start)) return nullptr;
  return a.devicePointer;
}

// One host <-> device copy of dsa_layer_step_host.
struct Copy {
  void* dst;
  const void* src;
  size_t bytes;
};

dsa_status check_step(const dsa_kv_layout* layout, const dsa_batch* batch, const void* q_idx, const float* w,
                      const void* q, int32_t topk, float sm_scale, const void* out, void* workspace,
                      size_t workspace_bytes, Ws& wl);
dsa_status run_step(const dsa_kv_layout* layout, const dsa_batch* batch, const void* q_idx, const float* w,
                    const void* q, int32_t topk, float sm_scale, int32_t* idx_out, void* out, float* lse,
                    void* workspace, const Ws& wl, dsa_stream_t stream);

}  // namespace

namespace dsa {
dsa_status record_cuda_status(cudaError_t e) { return cuda_status(e); }

// The CUDA context current on this thread (null before the runtime made one).
void* current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(p);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// cudaFuncSetAttribute(fn, attr, value) once per context: a kernel's attributes
// belong to the module loaded in a context, so another device (or a context made
// after a device reset) needs them set again.
cudaError_t set_func_attr_once(const void* fn, cudaFuncAttribute attr, int value) {
  struct Done {
    void* ctx;
    const void* fn;
    int attr, value;
  };
  static std::mutex mu;
  static std::vector<Done> done;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx)
    for (const Done& d : done)
      if (d.ctx == ctx && d.fn == fn && d.attr == static_cast<int>(attr) && d.value == value) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, attr, value);
  if (e == cudaSuccess) {
    ctx = current_context();   // made by the call above if there was none
    if (ctx) done.push_back({ctx, fn, static_cast<int>(attr), value});
  }
  return e;
}

// The argument checks of dsa_topk, shared with dsa_topk_noalloc.
dsa_status validate_topk_args(const dsa_kv_layout* layout, const dsa_batch* batch, const float* scores,
                              int64_t ld_scores, int32_t topk, const int32_t* idx, const int32_t* phys_slots) {
  dsa_status s;
  if (phys_slots && (s = check_layout(layout, false)) != DSA_OK) return s;
  if ((s = check_batch(batch, layout ? layout->block_size : 0)) != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_INVALID_ARG;
  if (batch->num_tokens > 0 && (!scores || !idx || !aligned16(scores))) return DSA_ERR_INVALID_ARG;
  if (ld_scores < batch->max_ctx_len || (ld_scores & 3)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}
}  // namespace dsa

extern "C" {

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

int32_t dsa_last_cuda_error(const char** name) {
  if (name) *name = g_last_cuda_name;
  return g_last_cuda;
}

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
  }
  return "DSA_ERR_UNKNOWN";
}

size_t dsa_workspace_size(const dsa_kv_layout* layout, const dsa_batch* batch, int32_t topk) {
  if (check_layout(layout, false) != DSA_OK) return 0;
  if (check_batch(batch, layout->block_size) != DSA_OK) return 0;
  if (topk < 1 || topk > DSA_MAX_TOPK) return 0;
  return plan_ws(layout, batch, topk).total;
}

dsa_status dsa_indexer_score(const dsa_kv_layout* layout, const dsa_batch* batch, const void* q_idx, const float* w,
                             float* scores, int64_t ld_scores, void* workspace, size_t workspace_bytes,
                             dsa_stream_t stream) {
  dsa_status s = check_layout(layout);
  if (s != DSA_OK) return s;
  if ((s = check_batch(batch, layout->block_size)) != DSA_OK) return s;
  if (batch->num_tokens > 0 && (!q_idx || !w || !scores || !aligned16(q_idx) || !aligned16(w) || !aligned16(scores)))
    return DSA_ERR_INVALID_ARG;
  if (ld_scores < batch->max_ctx_len || (ld_scores & 3)) return DSA_ERR_INVALID_ARG;
  if ((s = check_qidx(layout, batch, q_idx)) != DSA_OK) return s;
  const Ws wl = plan_ws(layout, batch, 1);
  if ((s = check_ws(workspace, workspace_bytes, wl)) != DSA_OK) return s;
  return run_indexer(layout, batch, q_idx, w, scores, ld_scores, workspace, wl, stream);
}

dsa_status dsa_topk(const dsa_kv_layout* layout, const dsa_batch* batch, const float* scores, int64_t ld_scores,
                    int32_t topk, int32_t* idx, int32_t* phys_slots, void* workspace, size_t workspace_bytes,
                    dsa_stream_t stream) {
  dsa_status s = validate_topk_args(layout, batch, scores, ld_scores, topk, idx, phys_slots);
  if (s != DSA_OK) return s;
  dsa_kv_layout dummy{};
  dummy.num_rows = 1;
  dummy.block_size = 64;
  const Ws wl = plan_ws(layout ? layout : &dummy, batch, topk);
  if ((s = check_ws(workspace, workspace_bytes, wl)) != DSA_OK) return s;
  return run_topk(layout, batch, scores, ld_scores, topk, idx, phys_slots, workspace, wl, stream, false);
}

dsa_status dsa_sparse_mla(const dsa_kv_layout* layout, const dsa_batch* batch, const void* q, const int32_t* idx,
                          int32_t topk, float sm_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                          dsa_stream_t stream) {
  dsa_status s = check_layout(layout);
  if (s != DSA_OK) return s;
  if ((s = check_batch(batch, layout->block_size)) != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK || !std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARG;
  if (batch->num_tokens > 0 && (!q || !idx || !out || !aligned16(q) || !aligned16(out))) return DSA_ERR_INVALID_ARG;
  const Ws wl = plan_ws(layout, batch, topk);
  if ((s = check_ws(workspace, workspace_bytes, wl)) != DSA_OK) return s;
  return run_mla(layout, batch, q, idx, nullptr, topk, sm_scale, out, lse, workspace, wl, stream, false);
}

dsa_status dsa_layer_step(const dsa_kv_layout* layout, const dsa_batch* batch, const void* q_idx, const float* w,
                          const void* q, int32_t topk, float sm_scale, int32_t* idx_out, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  Ws wl;
  const dsa_status s = check_step(layout, batch, q_idx, w, q, topk, sm_scale, out, workspace, workspace_bytes, wl);
  if (s != DSA_OK) return s;
  return run_step(layout, batch, q_idx, w, q, topk, sm_scale, idx_out, out, lse, workspace, wl, stream);
}

dsa_status dsa_layer_step_host(const dsa_kv_layout* layout, const dsa_batch* batch, void* q_idx, float* w, void* q,
                               int32_t topk, float sm_scale, int32_t* idx_out, void* out, float* lse,
                               const dsa_host_io* host, void* workspace, size_t workspace_bytes,
                               dsa_stream_t stream) {
  Ws wl;
  dsa_status s = check_step(layout, batch, q_idx, w, q, topk, sm_scale, out, workspace, workspace_bytes, wl);
  if (s != DSA_OK) return s;
  const int64_t T = batch->num_tokens, B = batch->num_reqs;
  if (!host || !host->ctx_lens || !host->block_table) return DSA_ERR_INVALID_ARG;
  if (T > 0 && (!host->q_idx || !host->w || !host->q || !host->q_req || !host->q_pos || !host->out))
    return DSA_ERR_INVALID_ARG;
  if ((host->lse && !lse) || (host->idx && !idx_out)) return DSA_ERR_INVALID_ARG;
  if (host->flags & ~DSA_HOST_PACKED) return DSA_ERR_INVALID_ARG;
  // in the order a packed layout follows
  const Copy in[7] = {
      {q, host->q, size_t(T) * kMlaHeads * kLatDim * 2},
      {q_idx, host->q_idx, q_idx_bytes(batch)},
      {w, host->w, size_t(T) * kIdxHeads * 4},
      {const_cast<int32_t*>(batch->q_req), host->q_req, size_t(T) * 4},
      {const_cast<int32_t*>(batch->q_pos), host->q_pos, size_t(T) * 4},
      {const_cast<int32_t*>(batch->ctx_lens), host->ctx_lens, size_t(B) * 4},
      {const_cast<int32_t*>(batch->block_table), host->block_table, size_t(B) * batch->bt_stride * 4},
  };
  const bool packed = (host->flags & DSA_HOST_PACKED) && T > 0;
  size_t total = in[0].bytes;
  if (packed)
    for (int i = 1; i < 7; ++i) {
      if (static_cast<const uint8_t*>(in[i].src) != static_cast<const uint8_t*>(in[0].src) + total ||
          static_cast<uint8_t*>(in[i].dst) != static_cast<uint8_t*>(in[0].dst) + total)
        return DSA_ERR_INVALID_ARG;
      total += in[i].bytes;
    }
  // page-locked ranges move in one copy kernel per direction (SM loads and stores
  // over the host link); other host memory through cudaMemcpyAsync
  const int nsm = num_sms();
  cudaError_t e = cudaSuccess;
  auto add = [&](HostCopyParams& hp, const Copy& c, bool to_host) {
    if (!c.bytes || e != cudaSuccess) return;
    void* m = mapped_device_ptr(to_host ? c.dst : c.src, c.bytes);
    if (m && hp.nseg < kHostCopyMaxSegs) {
      hp.seg[hp.nseg++] = {static_cast<uint8_t*>(to_host ? m : c.dst),
                           static_cast<const uint8_t*>(to_host ? c.src : m), c.bytes};
      return;
    }
    e = cudaMemcpyAsync(c.dst, c.src, c.bytes, to_host ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice, stream);
  };
  HostCopyParams hin{};
  if (packed) {
    add(hin, {in[0].dst, in[0].src, total}, false);
  } else {
    for (int i = 0; i < 7; ++i) add(hin, in[i], false);
  }
  // chained: its dependency wait covers the kernels before it; the scorer's set-up overlaps it
  if (e == cudaSuccess && hin.nseg) e = launch_host_copy(hin, nsm, stream, true);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((s = run_step(layout, batch, q_idx, w, q, topk, sm_scale, idx_out, out, lse, workspace, wl, stream)) != DSA_OK)
    return s;
  const Copy back[3] = {
      {host->out, out, size_t(T) * kMlaHeads * kVDim * 2},
      {host->lse, lse, host->lse ? size_t(T) * kMlaHeads * 4 : 0},
      {host->idx, idx_out, host->idx ? size_t(T) * size_t(topk) * 4 : 0},
  };
  HostCopyParams hout{};
  for (int i = 0; i < 3; ++i) add(hout, back[i], true);
  if (e == cudaSuccess && hout.nseg) e = launch_host_copy(hout, nsm, stream, true);
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

dsa_status check_step(const dsa_kv_layout* layout, const dsa_batch* batch, const void* q_idx, const float* w,
                      const void* q, int32_t topk, float sm_scale, const void* out, void* workspace,
                      size_t workspace_bytes, Ws& wl) {
  dsa_status s = check_layout(layout);
  if (s != DSA_OK) return s;
  if ((s = check_batch(batch, layout->block_size)) != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK || !std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARG;
  if (batch->num_tokens > 0 && (!q_idx || !w || !q || !out || !aligned16(q_idx) || !aligned16(w) ||
                                !aligned16(q) || !aligned16(out)))
    return DSA_ERR_INVALID_ARG;
  if ((s = check_qidx(layout, batch, q_idx)) != DSA_OK) return s;
  wl = plan_ws(layout, batch, topk);
  return check_ws(workspace, workspace_bytes, wl);
}

dsa_status run_step(const dsa_kv_layout* layout, const dsa_batch* batch, const void* q_idx, const float* w,
                    const void* q, int32_t topk, float sm_scale, int32_t* idx_out, void* out, float* lse,
                    void* workspace, const Ws& wl, dsa_stream_t stream) {
  dsa_status s;
  float* scores = at<float>(workspace, wl.scores);
  int32_t* idx = idx_out ? idx_out : at<int32_t>(workspace, wl.idx);
  // rows that the one-launch top-k takes start from the scorer's top-digit histograms
  uint32_t* row_hist = batch->max_ctx_len <= kTopkClusterMaxRow ? at<uint32_t>(workspace, wl.row_hist) : nullptr;
  // with FP8 latents the scorer also prepares the attention's query terms
  const bool fp8 = use_fp8_mla(wl);
  // rows beyond the one-launch top-k take three passes whose scratch must start at
  // zero: cleared before the scorer, so the passes follow the scorer directly
  const bool long_rows = batch->max_ctx_len > kTopkClusterMaxRow && batch->num_tokens > 0;
  if (long_rows) {
    const TopkScratch L = topk_scratch_layout(batch->num_tokens, wl.topk_nchunks);
    const cudaError_t e = cudaMemsetAsync(at<uint8_t>(workspace, wl.topk) + L.hist, 0, L.zero_end - L.hist, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if ((s = run_indexer(layout, batch, q_idx, w, scores, wl.ld, workspace, wl, stream, row_hist,
                       fp8 ? q : nullptr)) != DSA_OK)
    return s;
  // the top-k also emits each selection's physical cache slot, which the attention gathers directly
  int32_t* phys = at<int32_t>(workspace, wl.phys);
  // the top-k and the attention start while their predecessor drains (programmatic launch)
  if ((s = run_topk(layout, batch, scores, wl.ld, topk, idx, phys, workspace, wl, stream, true, row_hist, long_rows)) !=
      DSA_OK)
    return s;
  return run_mla(layout, batch, q, idx, phys, topk, sm_scale, out, lse, workspace, wl, stream, true, fp8);
}

}  // namespace

extern "C" {

dsa_status dsa_indexer_front(const dsa_kv_layout* layout, const dsa_batch* batch, const void* c_q, int32_t d_q,
                             const void* norm_weight, float eps, const void* w_qi, const float* head_w,
                             const void* k_new, void* q_idx, float* w_out, void* workspace, size_t workspace_bytes,
                             dsa_stream_t stream) {
  dsa_status s = check_layout(layout);
  if (s != DSA_OK) return s;
  if ((s = check_batch(batch, layout->block_size)) != DSA_OK) return s;
  if (d_q < 64 || d_q > 4096 || (d_q & 7) || !std::isfinite(eps) || eps < 0.f) return DSA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) || workspace_bytes < kStatusBytes)
    return DSA_ERR_WORKSPACE;
  const int T = batch->num_tokens;
  if (T == 0) return DSA_OK;
  if (!c_q || !norm_weight || !w_qi || !head_w || !q_idx || !w_out || !aligned16(c_q) || !aligned16(norm_weight) ||
      !aligned16(w_qi) || !aligned16(q_idx) || !aligned16(head_w) || !aligned16(w_out) || (k_new && !aligned16(k_new)))
    return DSA_ERR_INVALID_ARG;
  if ((s = check_qidx(layout, batch, q_idx)) != DSA_OK) return s;
  FrontParams p;
  p.b = batch_view(batch);
  p.pool = pool_view(layout);
  p.c_q = static_cast<const __nv_bfloat16*>(c_q);
  p.gamma = static_cast<const __nv_bfloat16*>(norm_weight);
  p.w_qi = static_cast<const __nv_bfloat16*>(w_qi);
  p.head_w = head_w;
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.q_idx = static_cast<uint8_t*>(q_idx);
  p.w_out = w_out;
  p.pool_w = static_cast<uint8_t*>(const_cast<void*>(layout->pool));
  p.d_q = d_q;
  p.eps = eps;
  p.status = static_cast<uint32_t*>(workspace);
  p.qmx = (batch->flags & DSA_BATCH_QIDX_MXFP4) ? 1 : 0;
  CUtensorMap wmap;
  if (!make_front_w_map(&wmap, w_qi, d_q)) return encode_fail();
  return cuda_status(launch_indexer_front(wmap, p, stream));
}

dsa_status dsa_write_latent(const dsa_kv_layout* layout, const dsa_batch* batch, const void* latent,
                            void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  dsa_status s = check_layout(layout);
  if (s != DSA_OK) return s;
  if ((s = check_batch(batch, layout->block_size)) != DSA_OK) return s;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) || workspace_bytes < kStatusBytes)
    return DSA_ERR_WORKSPACE;
  if (batch->num_tokens == 0) return DSA_OK;
  if (!latent || !aligned16(latent)) return DSA_ERR_INVALID_ARG;
  LatentWriteParams p;
  p.b = batch_view(batch);
  p.pool = pool_view(layout);
  p.latent = static_cast<const __nv_bfloat16*>(latent);
  p.pool_w = static_cast<uint8_t*>(const_cast<void*>(layout->pool));
  p.status = static_cast<uint32_t*>(workspace);
  return cuda_status(launch_write_latent(p, stream));
}

dsa_status dsa_check(void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  if (!workspace || workspace_bytes < kStatusBytes) return DSA_ERR_WORKSPACE;
  uint32_t word = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  if (word == 0) return DSA_OK;
  if ((e = cudaMemset(workspace, 0, sizeof(word))) != cudaSuccess) return cuda_fail(e);
  if (word & DEV_TIMEOUT) return DSA_ERR_TIMEOUT;
  return DSA_ERR_DEVICE_CHECK;
}

}  // extern "C"

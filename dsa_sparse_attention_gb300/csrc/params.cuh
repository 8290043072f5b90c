// params.cuh — kernel parameter blocks and launcher declarations.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace dsa {

struct IndexerParams {
  PoolView pool;
  BatchView b;
  const float* w;          // [T, 32]
  float* scores;           // [T, ld]
  int64_t ld;
  const PlanHeader* hdr;
  const ScoreGroup* groups;
  uint32_t* status;
  int direct;              // 1: one token per group, planned inside the scorer (hdr/groups unused)
  uint32_t* row_hist;      // [T, 2048] or null: per-token counts of the scores' top 11 key bits are
                           // added here (one token per group only); a hint for the top-k
  const __nv_bfloat16* mla_q = nullptr;   // [T, 96, 576] or null: in a layer step whose attention runs on
  uint8_t* mla_q_terms = nullptr;         // FP8 latents, the epilogue warps also write its query terms here
  int qmx = 0;                            // 1: MXFP4 queries (MXFP4 keys only): codes through the query map,
  const uint8_t* q_scales = nullptr;      //    and their E8M0 exponents [T, 32, 4] here
};

struct TopkParams {
  BatchView b;
  const float* scores;
  int64_t ld;
  int k;
  int chunk;            // scores per CTA (4096)
  int nchunks;          // chunks per row at max_ctx_len
  uint32_t* hist;       // [T, 2048]  top-digit histogram                 (zeroed)
  uint32_t* done;       // [T, 2]     per-pass CTA tickets                 (zeroed)
  uint32_t* cand_count; // [T]        candidates appended                  (zeroed)
  uint32_t* taken;      // [T, nchunks] candidates taken per chunk         (zeroed)
  uint32_t* thr;        // [T, 4]     digit b1, count above b1, key T, position cut
  uint32_t* gt;         // [T, nchunks] keys above digit b1 per chunk
  uint2* cands;         // [T, cap]   (key, position) in digit b1
  int cap;
  void* zero_begin;     // the zeroed fields are one contiguous region
  size_t zero_bytes;
  int32_t* idx;         // [T, k]
  int32_t* phys;        // [T, k] or null
  int log2_bs;
  uint32_t* status;
  uint32_t* pre_hist;   // [T, 2048] or null: top-digit counts left by the scorer (a hint, verified
                        // before use); the cluster top-k zeroes each row after reading it
};

struct MlaParams {
  PoolView pool;
  BatchView b;
  const __nv_bfloat16* q;  // [T, 96, 576] (read directly by the FP8 kernel)
  const int32_t* idx;      // [T, topk]
  const int32_t* phys;     // [T, topk] physical slots (row * bs + slot) of idx, or null
  int topk;
  float scale_log2;        // sm_scale * log2(e)
  int tps;                 // tiles per split
  int nsplit;
  __nv_bfloat16* out;      // [T, 96, 512]       (nsplit == 1)
  float* lse;              // [T, 96] or null    (nsplit == 1)
  __half* part_o;          // [T, nsplit, 512, 96] (nsplit > 1), dim-major, each normalised by its own sum
  float2* part_ml;         // [T, nsplit, 96]      (nsplit > 1): (max in log2 units, sum)
  const uint8_t* q_terms = nullptr;   // FP8 kernel: [T] query terms (mla_q.cuh layout)
  uint32_t* status;
};

constexpr int kTopkChunk = 4096;   // scores per CTA in the top-k passes
constexpr int kTopkClusterMaxRow = 65536;   // rows up to this long take the one-launch cluster top-k
// Decode batches of at most this many tokens, one per group, are planned inside
// the scorer (no separate planning launch).
constexpr int kDirectMaxT = 128;
constexpr int kTopkCap = 4096;     // candidates per row kept for the exact resolution

// Byte offsets of the top-k scratch inside a region (256-byte aligned segments);
// [hist .. zero_end) must be zeroed before the passes (launch_topk does it).
struct TopkScratch {
  size_t hist, done, cand_count, taken, zero_end, thr, gt, cands, total;
};

inline TopkScratch topk_scratch_layout(int64_t T, int nchunks) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  TopkScratch L;
  size_t off = 0;
  L.hist = off;
  off += size_t(T) * 2048 * 4;
  L.done = off;
  off += size_t(T) * 2 * 4;
  L.cand_count = off;
  off += size_t(T) * 4;
  L.taken = off;
  off += size_t(T) * nchunks * 4;
  L.zero_end = off;
  off = up(off);
  L.thr = off;
  off = up(off + size_t(T) * 4 * 4);
  L.gt = off;
  off = up(off + size_t(T) * nchunks * 4);
  L.cands = off;
  off = up(off + size_t(T) * kTopkCap * 8);
  L.total = off;
  return L;
}

inline void topk_bind_scratch(TopkParams& p, uint8_t* base, const TopkScratch& L, int nchunks) {
  p.chunk = kTopkChunk;
  p.nchunks = nchunks;
  p.hist = reinterpret_cast<uint32_t*>(base + L.hist);
  p.done = reinterpret_cast<uint32_t*>(base + L.done);
  p.cand_count = reinterpret_cast<uint32_t*>(base + L.cand_count);
  p.taken = reinterpret_cast<uint32_t*>(base + L.taken);
  p.thr = reinterpret_cast<uint32_t*>(base + L.thr);
  p.gt = reinterpret_cast<uint32_t*>(base + L.gt);
  p.cands = reinterpret_cast<uint2*>(base + L.cands);
  p.cap = kTopkCap;
  p.zero_begin = base + L.hist;
  p.zero_bytes = L.zero_end - L.hist;
}

// Launches `kern` on `st`; `chained` allows it to start before the previous
// kernel on the stream ends (it then calls grid_dep_wait before it reads that
// kernel's output), `cluster_x` > 0 groups its CTAs in clusters of that size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             bool chained, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  unsigned na = 0;
  if (chained) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster_x > 0) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = cluster_x;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The fused indexer front and the latent write (front.cu).
struct FrontParams {
  BatchView b;
  PoolView pool;
  const __nv_bfloat16* c_q;    // [T, d_q]
  const __nv_bfloat16* gamma;  // [d_q]
  const __nv_bfloat16* w_qi;   // [4096, d_q]
  const float* head_w;         // [T, 32]
  const __nv_bfloat16* k_new;  // [T, 128] or null
  uint8_t* q_idx;              // [T, 32, 128] e4m3
  float* w_out;                // [T, 32]
  uint8_t* pool_w;             // the pool, written at the new tokens' slots
  int d_q;
  float eps;
  uint32_t* status;
  int qmx = 0;                 // 1: q_idx in MXFP4 (codes [T, 32, 64], then E8M0 [T, 32, 4]), w_out = head_w
};

struct LatentWriteParams {
  BatchView b;
  PoolView pool;
  const __nv_bfloat16* latent;   // [T, 576]
  uint8_t* pool_w;
  uint32_t* status;
};

cudaError_t launch_indexer_front(const CUtensorMap& wmap, const FrontParams& p, cudaStream_t st);
cudaError_t launch_write_latent(const LatentWriteParams& p, cudaStream_t st);

// Host helpers (capi.cu): the CUDA context current on this thread, and
// cudaFuncSetAttribute done once per (context, kernel, attribute, value).
void* current_context();
cudaError_t set_func_attr_once(const void* fn, cudaFuncAttribute attr, int value);

cudaError_t launch_plan_groups(const BatchView& b, int G, ScoreGroup* groups, PlanHeader* hdr, uint32_t* status,
                               cudaStream_t st);
cudaError_t launch_indexer(const CUtensorMap& kmap, const CUtensorMap& qmap, const IndexerParams& p, int G,
                           int grid, cudaStream_t st);
int indexer_group_size(int idx_fmt, bool one_token_per_request);
// `zeroed`: the scratch [hist .. zero_end) was cleared on the stream already
// (otherwise the launch clears it first).
cudaError_t launch_topk(const TopkParams& p, cudaStream_t st, bool chained, bool zeroed = false);
cudaError_t launch_sparse_mla(const CUtensorMap& qmap, const CUtensorMap& cmap, const MlaParams& p, cudaStream_t st,
                              bool chained);
// FP8 latents, one 128-token tile per CTA (p.nsplit = tiles of the selection, p.tps
// = 1), followed by the split combine: whether it can run here, and the launch.
bool sparse_mla_fp8_available();
cudaError_t launch_sparse_mla_fp8(const CUtensorMap& pmap, const CUtensorMap& cmap, const MlaParams& p, cudaStream_t st,
                                  bool chained);
// The log-sum-exp merge of p.nsplit normalised partials into p.out / p.lse.
cudaError_t launch_mla_combine(const CUtensorMap& cmap, const MlaParams& p, cudaStream_t st);
// The query terms of a batch for the FP8 attention (a standalone call; a layer step's scorer writes them).
cudaError_t launch_mla_qprep(const __nv_bfloat16* q, uint8_t* terms, int T, cudaStream_t st);

}  // namespace dsa

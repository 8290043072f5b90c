// topk_noalloc.cu — dsa_topk for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside a CUDA
// stream callback or a host function node, plugins whose host framework owns
// every allocation and hands out none, or hard real-time loops that forbid any
// allocator traffic after start-up.  They cannot provide the workspace that
// dsa_topk needs for its per-query histograms and per-chunk counts.  This
// variant keeps that scratch in a fixed array in the library's own device
// memory instead, so the caller passes only the inputs and outputs.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds its DSA_NOALLOC_SCRATCH_BYTES until the process exits.  Host
// code cannot use the array's name as a device address, so the first call in
// each CUDA context looks the address up with cudaGetSymbolAddress (with that
// context's device current) and caches it under that context; that first call
// should therefore happen before any stream capture.  A context made later (a
// new device, or the primary context re-created after a device reset) gets its
// own lookup.  All calls share the one array and it keeps the last call's
// contents: the histograms are cleared on the stream at the start of every
// call that uses them, and two calls that overlap on the GPU (different
// streams, or concurrent host threads) race on it, so issue them in order on
// one stream.  Rows of at most 65,536 scores take the one-launch cluster
// kernel, which needs no global scratch; only longer rows use the array.
#include <mutex>
#include <vector>

#include "../../include/dsa.h"
#include "params.cuh"

namespace dsa {
dsa_status record_cuda_status(cudaError_t e);   // capi.cu: DSA_OK, or DSA_ERR_CUDA with the error recorded
dsa_status validate_topk_args(const dsa_kv_layout* layout, const dsa_batch* batch, const float* scores,
                              int64_t ld_scores, int32_t topk, const int32_t* idx, const int32_t* phys_slots);
}  // namespace dsa

namespace {

constexpr size_t kNoAllocBytes = DSA_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusBytes = 256;

static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocBytes];

std::mutex g_mu;
struct Entry {
  void* ctx;
  void* ptr;
};
std::vector<Entry> g_addr;   // device address of g_topk_scratch per CUDA context

// Device address of g_topk_scratch in the current context (looked up once per context).
cudaError_t scratch_address(void** out) {
  *out = nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  void* ctx = dsa::current_context();
  if (ctx)
    for (const Entry& e : g_addr)
      if (e.ctx == ctx) {
        *out = e.ptr;
        return cudaSuccess;
      }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
  if (e != cudaSuccess) return e;
  ctx = dsa::current_context();   // the runtime has made the context by now
  if (ctx) g_addr.push_back({ctx, p});
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" dsa_status dsa_topk_noalloc(const dsa_kv_layout* layout, const dsa_batch* batch, const float* scores,
                                       int64_t ld_scores, int32_t topk, int32_t* idx, int32_t* phys_slots,
                                       dsa_stream_t stream) {
  using namespace dsa;
  dsa_status s = validate_topk_args(layout, batch, scores, ld_scores, topk, idx, phys_slots);
  if (s != DSA_OK) return s;
  const int T = batch->num_tokens;
  if (T == 0) return DSA_OK;

  // scratch: the status word, then (rows over 65,536 scores only) the top-k
  // histograms, tickets, counts and candidates
  const int nchunks = static_cast<int>((batch->max_ctx_len + kTopkChunk - 1) / kTopkChunk);
  const TopkScratch L = topk_scratch_layout(T, nchunks);
  if (batch->max_ctx_len > kTopkClusterMaxRow && kStatusBytes + L.total > kNoAllocBytes)
    return DSA_ERR_WORKSPACE;   // batch too large for the fixed scratch

  void* addr = nullptr;
  const cudaError_t e = scratch_address(&addr);
  if (e != cudaSuccess) return record_cuda_status(e);
  uint8_t* base = static_cast<uint8_t*>(addr);

  int log2_bs = 0;
  if (layout)
    while ((1 << log2_bs) < layout->block_size) ++log2_bs;
  TopkParams p;
  p.b.T = T;
  p.b.B = batch->num_reqs;
  p.b.q_req = batch->q_req;
  p.b.q_pos = batch->q_pos;
  p.b.ctx_lens = batch->ctx_lens;
  p.b.bt = batch->block_table;
  p.b.bt_stride = batch->bt_stride;
  p.b.max_ctx = static_cast<int32_t>(batch->max_ctx_len);
  p.scores = scores;
  p.ld = ld_scores;
  p.k = topk;
  topk_bind_scratch(p, base + kStatusBytes, L, nchunks);
  p.idx = idx;
  p.phys = phys_slots;
  p.log2_bs = log2_bs;
  p.status = reinterpret_cast<uint32_t*>(base);
  p.pre_hist = nullptr;
  return record_cuda_status(launch_topk(p, stream, false));
}

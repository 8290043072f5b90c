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
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; that first call should therefore happen before any
// stream capture.  All calls share the one array and it keeps the last call's
// contents: the histograms are cleared on the stream at the start of every
// call, and two calls that overlap on the GPU (different streams, or
// concurrent host threads) race on it, so issue them in order on one stream.
#include <mutex>

#include "../../include/dsa.h"
#include "params.cuh"

namespace dsa {
dsa_status record_cuda_status(cudaError_t e);   // capi.cu: DSA_OK, or DSA_ERR_CUDA with the error recorded
}

namespace {

constexpr size_t kNoAllocBytes = DSA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_topk_scratch on the current device (looked up once).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" dsa_status dsa_topk_noalloc(const dsa_kv_layout* layout, const dsa_batch* batch, const float* scores,
                                       int64_t ld_scores, int32_t topk, int32_t* idx, int32_t* phys_slots,
                                       dsa_stream_t stream) {
  using namespace dsa;
  if (!batch || batch->num_tokens < 0 || batch->num_reqs < 1 || batch->bt_stride < 1 ||
      (batch->flags & ~DSA_BATCH_INVARIANT) || !batch->ctx_lens || !batch->block_table)
    return DSA_ERR_INVALID_ARG;
  if (batch->max_ctx_len < 1 || batch->max_ctx_len > (int64_t(1) << 30)) return DSA_ERR_INVALID_ARG;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_INVALID_ARG;
  int log2_bs = 0;
  if (phys_slots) {
    const int bs = layout ? layout->block_size : 0;
    if (bs < 16 || bs > 256 || (bs & (bs - 1))) return layout ? DSA_ERR_UNSUPPORTED : DSA_ERR_INVALID_ARG;
    if (batch->max_ctx_len > int64_t(batch->bt_stride) * bs) return DSA_ERR_INVALID_ARG;
    while ((1 << log2_bs) < bs) ++log2_bs;
  }
  if (ld_scores < batch->max_ctx_len || (ld_scores & 3)) return DSA_ERR_INVALID_ARG;
  const int T = batch->num_tokens;
  if (T == 0) return DSA_OK;
  if (!batch->q_req || !batch->q_pos || !scores || !idx || (reinterpret_cast<uintptr_t>(scores) & 15))
    return DSA_ERR_INVALID_ARG;

  // scratch: the status word, then the top-k histograms, tickets, counts and candidates
  const int nchunks = static_cast<int>((batch->max_ctx_len + kTopkChunk - 1) / kTopkChunk);
  const TopkScratch L = topk_scratch_layout(T, nchunks);
  if (256 + L.total > kNoAllocBytes) return DSA_ERR_WORKSPACE;   // batch too large for the fixed scratch

  uint8_t* base = static_cast<uint8_t*>(scratch_address());
  if (!base) return record_cuda_status(cudaErrorInvalidSymbol);

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
  topk_bind_scratch(p, base + 256, L, nchunks);
  p.idx = idx;
  p.phys = phys_slots;
  p.log2_bs = log2_bs;
  p.status = reinterpret_cast<uint32_t*>(base);
  p.pre_hist = nullptr;
  return record_cuda_status(launch_topk(p, stream, false));
}

// common.cuh — structures and helpers shared by the DSA kernels and the C ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace dsa {

constexpr int kIdxHeads = 32;
constexpr int kIdxDim = 128;
constexpr int kMlaHeads = 96;
constexpr int kLatDim = 576;
constexpr int kVDim = 512;
constexpr int kMaxTopk = 2048;
constexpr int kKeyTile = 128;   // keys per indexer MMA tile (M)
constexpr int kSelTile = 128;   // selected tokens per MLA tile (M of QK^T)

// Device view of the packed pool (one DSA layer).
struct PoolView {
  const uint8_t* pool;
  int64_t num_rows;
  int64_t row_stride;
  int64_t idx_off;
  int64_t lat_off;
  int32_t bs;
  int32_t log2_bs;
  int32_t idx_fmt;
  int32_t lat_fmt;
};

// Device view of the query batch.
struct BatchView {
  int32_t T;
  int32_t B;
  const int32_t* q_req;
  const int32_t* q_pos;
  const int32_t* ctx_lens;
  const int32_t* bt;
  int32_t bt_stride;
  int32_t max_ctx;   // host bound of ctx_lens (<= bt_stride * bs)
};

// A group of consecutive query tokens of one request that share every key tile.
struct ScoreGroup {
  int32_t t0;          // first token
  int32_t n;           // tokens in the group (1..G)
  int32_t req;         // request
  int32_t L;           // keys to score = 1 + max position in the group
  int32_t tile_begin;  // first global key-tile index of the group
  int32_t pad[3];
};

struct PlanHeader {
  int32_t n_groups;
  int32_t total_tiles;
  int32_t pad[6];
};

// Request / position of token t, clamped into range; out-of-range inputs are
// recorded in the status word so no kernel reads outside its buffers.
__device__ __forceinline__ void load_token(const BatchView& b, int t, uint32_t* status, int& req, int& pos) {
  int r = b.q_req[t];
  int p = b.q_pos[t];
  bool bad = false;
  if (r < 0 || r >= b.B) { bad = true; r = r < 0 ? 0 : b.B - 1; }
  int L = b.ctx_lens[r];
  if (L > b.max_ctx || L < 1) { bad = true; L = L < 1 ? 1 : b.max_ctx; }
  if (p < 0 || p >= L) { bad = true; p = p < 0 ? 0 : L - 1; }
  if (bad) atomicOr(status, DEV_BAD_BATCH);
  req = r;
  pos = p;
}

// Order-preserving map of a float score to uint32 (larger float -> larger key);
// -0.0 is folded onto +0.0 first so the two compare equal.
__device__ __forceinline__ uint32_t score_key(float f) {
  f = f + 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ constexpr int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace dsa

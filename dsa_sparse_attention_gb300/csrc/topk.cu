// topk.cu — exact per-query top-k over fp32 scores by radix selection.
//
// vLLM K3.1 Pro day-0 post, "Sparse Attention in K3.1 Pro": the indexer keeps
// the top 2,048 tokens and attention runs exactly over them; "An exact top-k
// merge with 10x less traffic" selects the global top-2048 with a radix select
// over a small candidate set, falling back to a full resend when the candidates
// do not suffice; "Zero-mismatch RL on day 0" asks for a top-k whose result does
// not depend on the batch.  Here, per query row of n scores split into chunks
// of 4096 (one CTA each, so a 1M-token row still spreads over 256 CTAs):
//  1. hist:       11-bit histogram of the top digit of each score's order-
//                 preserving key; the last CTA of the row finds the digit b1 that
//                 holds the k-th largest key and the count above it.
//  2. candidates: each chunk counts its keys above digit b1 and appends the keys
//                 in digit b1 (the candidates) to a per-row list; then one CTA
//                 of 1,024 threads per row resolves the exact threshold key T
//                 among them, and the position cut for keys equal to T (lowest
//                 positions first), then counts per chunk how many candidates
//                 are taken.  If the list overflows (heavy ties), that CTA
//                 redoes this step exactly over the whole row.
//  3. emit:       ordered compaction: chunk c writes its selected positions after
//                 those of chunks < c, so the output is ascending, deterministic
//                 and independent of the rest of the batch.
// Rows of at most 65,536 scores take a one-launch path instead: a cluster of up
// to eight CTAs per row keeps the row in registers (16 scores per thread).  The
// top digit's histogram comes from the scorer (inside a layer step, verified by
// exact counts) or is merged through distributed shared memory; each CTA then
// lists its keys in the threshold digit, every CTA gathers the row's list and
// resolves the remaining two digits (11 + 10 bits) and the position cut locally,
// and each CTA writes its selections after those of the CTAs before it.  Heavy
// ties (more than 4,096 keys in the threshold digit) resolve the two digits
// through the cluster instead.  No global scratch (the hint histograms are left
// zeroed for the next layer step).
#include "params.cuh"

namespace dsa {

constexpr int kTopkThreads = 256;
constexpr int kBins = 2048;
constexpr int kPerThread = 16;                       // scores per thread per chunk
static_assert(kTopkThreads * kPerThread == 4096, "chunk");
static_assert(kTopkCap <= 4096, "the resolving CTA stages the candidate list in its 4096-entry buffer");

// Order of the 16 scores a thread owns in its chunk: [c0 + 16*tid, +16).
__device__ __forceinline__ void load16(const float* row, int s0, int c1, uint32_t (&u)[kPerThread]) {
  if (s0 + kPerThread <= c1) {
    const float4* p4 = reinterpret_cast<const float4*>(row + s0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldcg(p4 + q);
      u[4 * q + 0] = score_key(v.x);
      u[4 * q + 1] = score_key(v.y);
      u[4 * q + 2] = score_key(v.z);
      u[4 * q + 3] = score_key(v.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) u[i] = (s0 + i < c1) ? score_key(__ldcg(row + s0 + i)) : 0u;
  }
}

// Block-wide exclusive scan of one uint32 per thread; also returns the total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* sh, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < nw ? sh[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;   // inclusive per warp
  }
  __syncthreads();
  total = sh[nw - 1];
  const uint32_t excl = (warp > 0 ? sh[warp - 1] : 0u) + x - v;
  __syncthreads();
  return excl;
}

// In a histogram of `nbins` bins ordered by key, the bin holding the kk-th
// largest element (1-based) and the number of elements in higher bins.
// `hist` may be shared or global memory.  Uses sh[0..40].
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t kk, int& bin, uint32_t& above, uint32_t* sh) {
  const int per = nbins / blockDim.x;
  const int hi = nbins - static_cast<int>(threadIdx.x) * per;
  uint32_t local = 0;
  for (int b = hi - 1; b >= hi - per; --b) local += hist[b];
  uint32_t total;
  const uint32_t excl = block_excl_scan(local, sh, total);
  if (excl < kk && excl + local >= kk) {
    uint32_t cum = excl;
    for (int b = hi - 1; b >= hi - per; --b) {
      const uint32_t h = hist[b];
      if (cum + h >= kk) {
        sh[33] = static_cast<uint32_t>(b);
        sh[34] = cum;
        break;
      }
      cum += h;
    }
  }
  __syncthreads();
  bin = static_cast<int>(sh[33]);
  above = sh[34];
  __syncthreads();
}

// Physical slot (row * block_size + slot) of position s.
__device__ __forceinline__ int32_t emit_phys(const TopkParams& p, const int32_t* btrow, int s, int bs_mask) {
  return (btrow[s >> p.log2_bs] << p.log2_bs) | (s & bs_mask);
}

__device__ __forceinline__ bool row_range(const TopkParams& p, int t, int& c0, int& c1, int& n) {
  int req, pos;
  load_token(p.b, t, p.status, req, pos);
  n = pos + 1;
  c0 = blockIdx.x * p.chunk;
  c1 = min(n, c0 + p.chunk);
  return c0 < n;
}

// The last CTA (by ticket) of row t to finish a pass; call with every thread.
__device__ __forceinline__ bool last_of_row(uint32_t* counter, int nchunks_row, uint32_t* sh) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh[40] = atomicAdd(counter, 1u);
  __syncthreads();
  const bool last = sh[40] == static_cast<uint32_t>(nchunks_row - 1);
  if (last) __threadfence();
  return last;
}

// ------------------------------------------------------------------- pass 1

__global__ void __launch_bounds__(kTopkThreads) topk_hist_kernel(TopkParams p) {
  __shared__ uint32_t h[kBins];
  __shared__ uint32_t sh[48];
  const int t = blockIdx.y;
  int c0, c1, n;
  const bool work = row_range(p, t, c0, c1, n) && n > p.k;   // inputs of the call, read before the wait
  grid_dep_wait();     // the scores (and the zeroed scratch) of the work before
  grid_dep_launch();
  if (!work) return;
  for (int i = threadIdx.x; i < kBins; i += kTopkThreads) h[i] = 0;
  __syncthreads();
  const float* row = p.scores + static_cast<int64_t>(t) * p.ld;
  uint32_t u[kPerThread];
  const int s0 = c0 + threadIdx.x * kPerThread;
  load16(row, s0, c1, u);
#pragma unroll
  for (int i = 0; i < kPerThread; ++i)
    if (s0 + i < c1) atomicAdd(&h[u[i] >> 21], 1u);
  __syncthreads();
  uint32_t* gh = p.hist + static_cast<int64_t>(t) * kBins;
  for (int i = threadIdx.x; i < kBins; i += kTopkThreads)
    if (h[i]) atomicAdd(gh + i, h[i]);
  const int nch = static_cast<int>(cdiv(n, p.chunk));
  if (!last_of_row(p.done + 2 * t, nch, sh)) return;
  for (int i = threadIdx.x; i < kBins; i += kTopkThreads) h[i] = __ldcg(gh + i);
  __syncthreads();
  int b1;
  uint32_t above;
  find_bin(h, kBins, static_cast<uint32_t>(p.k), b1, above, sh);
  if (threadIdx.x == 0) {
    p.thr[4 * t + 0] = static_cast<uint32_t>(b1);
    p.thr[4 * t + 1] = above;
  }
}

// ------------------------------------------------------------------- pass 2

// Exact resolution of the threshold among keys with top digit b1, by one CTA.
// Inputs either the candidate list (smem-resident) or, on overflow, the row.
struct Resolve {
  uint32_t T;        // threshold key
  int32_t cut;       // keys == T are taken at positions <= cut
};

// Returns the kk-th largest value (1-based) of the 21-bit low parts of the
// elements produced by `gen(i, key, idx, valid)` for i < count, and the number
// of elements strictly above it.  Two digit passes: 11 + 10 bits.
template <typename Gen>
__device__ void select_low21(Gen gen, int count, uint32_t kk, uint32_t& value, uint32_t& above, uint32_t* h,
                             uint32_t* sh) {
  // pass A: bits 20..10
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < count; i += blockDim.x) {
    uint32_t key;
    int32_t idx;
    if (gen(i, key, idx)) atomicAdd(&h[(key >> 10) & 2047u], 1u);
  }
  __syncthreads();
  int bA;
  uint32_t aA;
  find_bin(h, kBins, kk, bA, aA, sh);
  // pass B: bits 9..0 among digit bA
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < count; i += blockDim.x) {
    uint32_t key;
    int32_t idx;
    if (gen(i, key, idx) && ((key >> 10) & 2047u) == static_cast<uint32_t>(bA)) atomicAdd(&h[key & 1023u], 1u);
  }
  __syncthreads();
  int bB;
  uint32_t aB;
  find_bin(h, 1024, kk - aA, bB, aB, sh);
  value = (static_cast<uint32_t>(bA) << 10) | static_cast<uint32_t>(bB);
  above = aA + aB;
}

// The m-th smallest position (1-based) among elements with key == T.
template <typename Gen>
__device__ int32_t select_cut(Gen gen, int count, uint32_t T, uint32_t m, uint32_t* h, uint32_t* sh) {
  // positions < 2^30: three 10-bit digits, smallest first = largest of (2^30-1-pos)
  uint32_t prefix = 0, got = 0;
  for (int level = 0; level < 3; ++level) {
    const int shift = 20 - 10 * level;
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) h[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < count; i += blockDim.x) {
      uint32_t key;
      int32_t idx;
      if (gen(i, key, idx) && key == T) {
        const uint32_t v = 0x3FFFFFFFu - static_cast<uint32_t>(idx);
        if (level == 0 || (v >> (shift + 10)) == prefix) atomicAdd(&h[(v >> shift) & 1023u], 1u);
      }
    }
    __syncthreads();
    int b;
    uint32_t a;
    find_bin(h, 1024, m - got, b, a, sh);
    prefix = (prefix << 10) | static_cast<uint32_t>(b);
    got += a;
  }
  return static_cast<int32_t>(0x3FFFFFFFu - prefix);
}

__global__ void __launch_bounds__(kTopkThreads) topk_candidates_kernel(TopkParams p) {
  __shared__ uint32_t sh[48];
  __shared__ uint32_t lcount, lbase;
  __shared__ uint2 lc[4096];       // this chunk's candidates (key, position)
  const int t = blockIdx.y;
  int c0, c1, n;
  const bool work = row_range(p, t, c0, c1, n) && n > p.k;
  grid_dep_wait();     // the histogram pass
  grid_dep_launch();
  if (!work) return;
  const uint32_t b1 = p.thr[4 * t + 0];
  const float* row = p.scores + static_cast<int64_t>(t) * p.ld;
  if (threadIdx.x == 0) lcount = 0;
  __syncthreads();
  uint32_t u[kPerThread];
  const int s0 = c0 + threadIdx.x * kPerThread;
  load16(row, s0, c1, u);
  uint32_t gt = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    if (s0 + i >= c1) continue;
    const uint32_t d = u[i] >> 21;
    gt += d > b1;
    if (d == b1) {
      const uint32_t slot = atomicAdd(&lcount, 1u);
      lc[slot] = make_uint2(u[i], static_cast<uint32_t>(s0 + i));
    }
  }
  uint32_t total;
  block_excl_scan(gt, sh, total);
  if (threadIdx.x == 0) {
    p.gt[static_cast<int64_t>(t) * p.nchunks + blockIdx.x] = total;
    lbase = atomicAdd(p.cand_count + t, lcount);
  }
  __syncthreads();
  uint2* cand = p.cands + static_cast<int64_t>(t) * p.cap;
  for (uint32_t i = threadIdx.x; i < lcount; i += kTopkThreads)
    if (lbase + i < static_cast<uint32_t>(p.cap)) cand[lbase + i] = lc[i];
}

// Exact resolution of each row's threshold among its candidates: one CTA of
// kResolveThreads per row, after every chunk of the row has listed its candidates.
constexpr int kResolveThreads = 1024;

__global__ void __launch_bounds__(kResolveThreads) topk_resolve_kernel(TopkParams p) {
  __shared__ uint32_t h[kBins];
  __shared__ uint32_t sh[48];
  __shared__ uint2 lc[4096];       // the row's candidates (key, position)
  const int t = blockIdx.x;
  int req, pos;
  load_token(p.b, t, p.status, req, pos);   // inputs of the call, read before the wait
  grid_dep_wait();     // the candidate pass
  grid_dep_launch();
  const int n = pos + 1;
  if (n <= p.k) return;
  const int nch = static_cast<int>(cdiv(n, p.chunk));
  const uint32_t b1 = p.thr[4 * t + 0];
  const float* row = p.scores + static_cast<int64_t>(t) * p.ld;
  const uint2* cand = p.cands + static_cast<int64_t>(t) * p.cap;
  const uint32_t r = static_cast<uint32_t>(p.k) - p.thr[4 * t + 1];   // to take from digit b1
  const uint32_t count = __ldcg(p.cand_count + t);
  uint32_t Tlow, aboveT;
  int32_t cut;
  uint32_t* taken = p.taken + static_cast<int64_t>(t) * p.nchunks;
  if (count <= static_cast<uint32_t>(p.cap)) {
    // the whole candidate list fits this CTA's staging buffer (cap == 4096)
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) lc[i] = __ldcg(cand + i);
    __syncthreads();
    auto gen = [&](int i, uint32_t& key, int32_t& idx) {
      const uint2 c = lc[i];
      key = c.x & 0x1FFFFFu;
      idx = static_cast<int32_t>(c.y);
      return true;
    };
    select_low21(gen, static_cast<int>(count), r, Tlow, aboveT, h, sh);
    // h still holds the last digit's counts: h[Tlow & 1023] keys equal T.  When all of
    // them are taken (the usual case) no position cut is needed.
    const uint32_t eq = h[Tlow & 1023u];
    cut = eq == r - aboveT ? 0x7FFFFFFF : select_cut(gen, static_cast<int>(count), Tlow, r - aboveT, h, sh);
    // selections per chunk: counted in shared memory (this CTA alone writes the row's
    // counts, which start at zero), or with global atomics for rows of more chunks
    const bool in_smem = nch <= kBins;
    if (in_smem) {
      __syncthreads();   // every thread is done reading h
      for (int c = threadIdx.x; c < nch; c += static_cast<int>(blockDim.x)) h[c] = 0;
      __syncthreads();
    }
    for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) {
      const uint2 c = lc[i];
      const uint32_t lo = c.x & 0x1FFFFFu;
      if (lo > Tlow || (lo == Tlow && static_cast<int32_t>(c.y) <= cut)) {
        const uint32_t ch = c.y / static_cast<uint32_t>(p.chunk);
        if (in_smem) atomicAdd(&h[ch], 1u);
        else atomicAdd(taken + ch, 1u);
      }
    }
    if (in_smem) {
      __syncthreads();
      for (int c = threadIdx.x; c < nch; c += static_cast<int>(blockDim.x))
        if (h[c]) taken[c] = h[c];
    }
  } else {
    // heavy ties: redo the resolution over the whole row in this CTA
    auto gen = [&](int i, uint32_t& key, int32_t& idx) {
      const uint32_t k = score_key(__ldcg(row + i));
      key = k & 0x1FFFFFu;
      idx = i;
      return (k >> 21) == b1;
    };
    select_low21(gen, n, r, Tlow, aboveT, h, sh);
    cut = select_cut(gen, n, Tlow, r - aboveT, h, sh);
    for (int i = threadIdx.x; i < n; i += static_cast<int>(blockDim.x)) {
      uint32_t key;
      int32_t idx;
      if (gen(i, key, idx) && (key > Tlow || (key == Tlow && idx <= cut)))
        atomicAdd(taken + i / p.chunk, 1u);
    }
  }
  if (threadIdx.x == 0) {
    p.thr[4 * t + 2] = (b1 << 21) | Tlow;
    p.thr[4 * t + 3] = static_cast<uint32_t>(cut);
  }
}

// ------------------------------------------------------------------- pass 3

__global__ void __launch_bounds__(kTopkThreads) topk_emit_kernel(TopkParams p) {
  __shared__ uint32_t sh[48];
  __shared__ uint32_t base_sh;
  const int t = blockIdx.y;
  int req, pos;
  load_token(p.b, t, p.status, req, pos);
  grid_dep_wait();     // the candidate pass
  grid_dep_launch();
  const int n = pos + 1;
  const int c0 = blockIdx.x * p.chunk;
  const int c1 = min(n, c0 + p.chunk);
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.k;
  int32_t* phys = p.phys ? p.phys + static_cast<int64_t>(t) * p.k : nullptr;
  const int32_t* btrow = p.b.bt + static_cast<int64_t>(req) * p.b.bt_stride;
  const int bs_mask = (1 << p.log2_bs) - 1;

  if (n <= p.k) {   // every position is selected; chunk 0 also writes the -1 tail
    for (int s = c0 + threadIdx.x; s < c1; s += kTopkThreads) {
      out[s] = s;
      if (phys) phys[s] = emit_phys(p, btrow, s, bs_mask);
    }
    if (blockIdx.x == 0)
      for (int s = n + threadIdx.x; s < p.k; s += kTopkThreads) {
        out[s] = -1;
        if (phys) phys[s] = -1;
      }
    return;
  }
  if (c0 >= n) return;
  const uint32_t T = __ldcg(p.thr + 4 * t + 2);
  const int32_t cut = static_cast<int32_t>(__ldcg(p.thr + 4 * t + 3));
  // positions selected by earlier chunks
  {
    uint32_t part = 0;
    const uint32_t* gt = p.gt + static_cast<int64_t>(t) * p.nchunks;
    const uint32_t* tk = p.taken + static_cast<int64_t>(t) * p.nchunks;
    for (int c = threadIdx.x; c < static_cast<int>(blockIdx.x); c += kTopkThreads) part += __ldcg(gt + c) + __ldcg(tk + c);
    uint32_t total;
    block_excl_scan(part, sh, total);
    if (threadIdx.x == 0) base_sh = total;
    __syncthreads();
  }
  const float* row = p.scores + static_cast<int64_t>(t) * p.ld;
  uint32_t u[kPerThread];
  const int s0 = c0 + threadIdx.x * kPerThread;
  load16(row, s0, c1, u);
  uint32_t mine = 0, flags = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int s = s0 + i;
    const bool take = s < c1 && (u[i] > T || (u[i] == T && s <= cut));
    flags |= static_cast<uint32_t>(take) << i;
    mine += take;
  }
  uint32_t total;
  uint32_t o = base_sh + block_excl_scan(mine, sh, total);
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    if (!((flags >> i) & 1u)) continue;
    const int s = s0 + i;
    if (o < static_cast<uint32_t>(p.k)) {
      out[o] = s;
      if (phys) phys[o] = emit_phys(p, btrow, s, bs_mask);
    }
    ++o;
  }
}

// ------------------------------------------------------- one-launch cluster path

constexpr int kClThreads = 512;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClSlice = kClThreads * kPerThread;   // 8192 scores per CTA
constexpr int kClMaxCtas = 8;                       // portable cluster size
constexpr int kClMaxRow = kClSlice * kClMaxCtas;    // 65,536
constexpr int kClOwn = kBins / 2;                   // bins a CTA owns when the cluster has >= 2 CTAs
constexpr int kClCap = 4096;                        // candidates of a row gathered into every CTA
constexpr int kClPer4 = (kClCap / 4 + kClMaxCtas + kClThreads - 1) / kClThreads;   // 16-byte groups per thread (padded lists)
static_assert(kClThreads * 4 == kBins, "one thread per four bins of the top digit");
static_assert(kClMaxRow == kTopkClusterMaxRow, "row limit of the cluster path");

struct ClShared {
  // zeroed at the start (the first six arrays, contiguous)
  uint32_t hl[kBins];             // this CTA's digit-1 histogram
  uint32_t hr[kClOwn];            // the digit-1 bins this CTA owns, summed over the cluster
  uint32_t h2[kBins];             // digit-2 histogram (of the row's candidates, or of this CTA's keys)
  uint32_t h3[1024];              // digit-3 histogram
  uint32_t hr2[kClOwn];           // owned digit-2 bins (many candidates)
  uint32_t hr3[kClOwn / 2];       // owned digit-3 bins (many candidates)
  uint32_t cl[kClCap];            // this CTA's candidate keys, in position order
  uint32_t wsh[8][32];            // scratch of the scans and searches, one row per call site
  uint32_t res[2];
  uint32_t meta[kClMaxCtas];      // per CTA: (keys above digit b1) << 16 | (keys in digit b1)
  uint32_t meta_b1[kClMaxCtas];   // per CTA: the digit b1 those counts refer to
  uint32_t counts[kClMaxCtas];    // per CTA: (keys above T) << 16 | (keys equal to T)
};
constexpr int kClZeroWords = kBins + kClOwn + kBins + 1024 + kClOwn + kClOwn / 2;

// Exclusive scan of one value per thread over the block with a single barrier:
// (this thread's exclusive prefix, block total); `wsh` must not be in use by
// another call until a later barrier.
__device__ __forceinline__ uint2 cl_excl_scan(uint32_t v, uint32_t* wsh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsh[warp] = x;
  __syncthreads();
  const uint32_t wv = lane < kClWarps ? wsh[lane] : 0u;
  return make_uint2(__reduce_add_sync(0xffffffffu, lane < warp ? wv : 0u) + x - v, __reduce_add_sync(0xffffffffu, wv));
}

// Exclusive scan of v over the block and block sums of x and y, with one barrier;
// `wa`, `wb`: two scratch rows (32 words each) not in use by another call until a
// later barrier.  Returns the scan; x and y become the sums.
__device__ __forceinline__ uint32_t cl_scan_sum2(uint32_t v, uint32_t& x, uint32_t& y, uint32_t* wa, uint32_t* wb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t s = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t z = __shfl_up_sync(0xffffffffu, s, o);
    if (lane >= o) s += z;
  }
  const uint32_t xs = __reduce_add_sync(0xffffffffu, x), ys = __reduce_add_sync(0xffffffffu, y);
  if (lane == 31) wa[warp] = s;
  if (lane == 0) {
    wb[warp] = xs;
    wb[kClWarps + warp] = ys;
  }
  __syncthreads();
  const uint32_t wv = lane < kClWarps ? wa[lane] : 0u;
  x = __reduce_add_sync(0xffffffffu, lane < kClWarps ? wb[lane] : 0u);
  y = __reduce_add_sync(0xffffffffu, lane < kClWarps ? wb[kClWarps + lane] : 0u);
  return __reduce_add_sync(0xffffffffu, lane < warp ? wv : 0u) + s - v;
}

// Thread i holds bins 4i .. 4i+3 (ascending key order) of a histogram.  Finds the
// bin holding the kk-th largest element (kk >= 1) and the number of elements in
// higher bins, as (bin, above); (~0u, 0) when the histogram holds fewer than kk.
// Two barriers.
__device__ __forceinline__ uint2 cl_find(uint4 c, uint32_t kk, uint32_t* wsh, uint32_t* res) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t s = c.x + c.y + c.z + c.w;
  uint32_t x = s;   // becomes the sum over lanes >= this one (higher bins)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) wsh[warp] = x;
  __syncthreads();
  const uint32_t wv = lane < kClWarps ? wsh[lane] : 0u;
  uint32_t cum = __reduce_add_sync(0xffffffffu, lane > warp ? wv : 0u) + x - s;
  const uint32_t total = __reduce_add_sync(0xffffffffu, wv);
  if (cum < kk && cum + s >= kk) {
    int b = 4 * static_cast<int>(threadIdx.x) + 3;
    if (cum + c.w < kk) {
      cum += c.w;
      --b;
      if (cum + c.z < kk) {
        cum += c.z;
        --b;
        if (cum + c.y < kk) {
          cum += c.y;
          --b;
        }
      }
    }
    res[0] = static_cast<uint32_t>(b);
    res[1] = cum;
  } else if (threadIdx.x == 0 && total < kk) {
    // fewer than kk elements (only a hint histogram can be short): no bin, ~0u
    res[0] = 0xFFFFFFFFu;
    res[1] = 0u;
  }
  __syncthreads();
  return make_uint2(res[0], res[1]);
}

// One CTA of a cluster of up to eight per query row; the row stays in registers
// (16 scores per thread).
//  1. Digit 1 (the top 11 key bits): with PRE, the histogram the scorer left for
//     the row; else each CTA's histogram, its non-empty bins added into the CTA
//     owning them (a contiguous 1/csize of the bins) through distributed shared
//     memory and read back four bins per thread.  The bin b1 holding the k-th key
//     follows.
//  2. Each CTA counts its keys above b1, lists its keys in b1 (the candidates) in
//     position order and publishes both counts to every CTA.  The counts decide
//     exactly whether b1 holds the k-th key; a hint that fails is replaced by the
//     histogram of step 1 built from the scores.
//  3. Up to kClCap candidates: every CTA gathers the row's candidates and resolves
//     digits 2 and 3 (bits 20..10, 9..0) locally.  More (heavy ties): digits 2 and
//     3 through the cluster as in step 1, over the keys in registers.
//  4. Ordered output: keys above the threshold key T, then keys equal to T at the
//     lowest positions, each CTA after the selections of the CTAs before it.
template <bool PRE>
__global__ void __launch_bounds__(kClThreads) topk_cluster_kernel(TopkParams p) {
  __shared__ __align__(16) ClShared S;
  const int t = blockIdx.y;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank(), csize = cluster_size();
  const bool multi = csize > 1;
  // Inputs of the call (not of the kernel before): the row length and the
  // block-table entry of this thread's 16 positions are read before the wait.
  int req, pos;
  load_token(p.b, t, p.status, req, pos);
  const int n = pos + 1;
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.k;
  int32_t* phys = p.phys ? p.phys + static_cast<int64_t>(t) * p.k : nullptr;
  const int32_t* btrow = p.b.bt + static_cast<int64_t>(req) * p.b.bt_stride;
  const int bs_mask = (1 << p.log2_bs) - 1;
  // this CTA's slice of the row, a multiple of 16 scores long (<= 8192)
  const int SL = (static_cast<int>(cdiv(n, csize)) + 15) & ~15;
  const int c0 = static_cast<int>(rank) * SL;
  const int c1 = min(n, c0 + SL);
  const int s0 = c0 + tid * kPerThread;
  const int nv = max(0, min(kPerThread, c1 - s0));
  // 16 consecutive positions from a multiple of 16 share one block when bs >= 16
  const bool one_block = p.log2_bs >= 4;
  const int32_t blk = (phys && one_block && nv > 0 && n > p.k) ? __ldcg(btrow + (s0 >> p.log2_bs)) : 0;
  for (int i = tid; i < kClZeroWords; i += kClThreads) S.hl[i] = 0;
  grid_dep_wait();
  grid_dep_launch();
  uint4* gh = PRE ? reinterpret_cast<uint4*>(p.pre_hist + static_cast<int64_t>(t) * kBins) : nullptr;

  if (n <= p.k) {   // every position is selected, then -1 padding
    for (int s = rank * kClThreads + tid; s < p.k; s += csize * kClThreads) {
      out[s] = s < n ? s : -1;
      if (phys) phys[s] = s < n ? emit_phys(p, btrow, s, bs_mask) : -1;
    }
    if (PRE && rank == 0) gh[tid] = make_uint4(0u, 0u, 0u, 0u);
    return;   // uniform over the cluster: no CTA touches another's shared memory
  }
  const float* row = p.scores + static_cast<int64_t>(t) * p.ld;
  uint4 c = make_uint4(0u, 0u, 0u, 0u);
  if (PRE) c = __ldcg(gh + tid);
  uint32_t u[kPerThread];
  load16(row, s0, s0 + nv, u);
  __syncthreads();   // zeroed
  bool pending = multi;
  // Every CTA has started (and zeroed) before any CTA writes into it.  With the hint
  // the first writes come after the publishing barrier, which orders the zeroing, so
  // this arrival is only a signal.
  if (multi) {
    if (PRE) cluster_arrive_relaxed();
    else cluster_arrive();
  }
  const uint32_t k = static_cast<uint32_t>(p.k);

  // ---- steps 1 and 2 (twice when a hint fails)
  int b1 = 0;
  uint32_t G = 0, Cc = 0;
  bool exchange = !PRE;
#pragma unroll 1
  for (int round = 0; round < 2; ++round) {
    if (exchange) {
#pragma unroll
      for (int i = 0; i < kPerThread; ++i)
        if (i < nv) atomicAdd(&S.hl[u[i] >> 21], 1u);
      __syncthreads();
      if (multi) {
        const uint32_t own = ((kBins + csize - 1) / csize + 3u) & ~3u;   // four-bin multiple: one owner per thread
        if (pending) {
          cluster_wait();
          pending = false;
        }
        for (int b = tid; b < kBins; b += kClThreads) {
          const uint32_t v = S.hl[b];
          if (v == 0) continue;
          const uint32_t o = static_cast<uint32_t>(b) / own;
          red_cluster_add(cluster_map(smem_u32(&S.hr[b - o * own]), o), v);
        }
        cluster_sync();
        const uint32_t b0 = 4u * tid, o = b0 / own;
        c = ld_cluster_v4(cluster_map(smem_u32(&S.hr[b0 - o * own]), o));
      } else {
        c = *reinterpret_cast<const uint4*>(&S.hl[4 * tid]);
      }
    }
    b1 = static_cast<int>(cl_find(c, k, S.wsh[0], S.res).x);
    uint32_t gtm = 0, cm = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const uint32_t d = u[i] >> 21;
      if (i < nv) {
        gtm |= static_cast<uint32_t>(d > static_cast<uint32_t>(b1)) << i;
        cm |= static_cast<uint32_t>(d == static_cast<uint32_t>(b1)) << i;
      }
    }
    const uint2 sc = cl_excl_scan((static_cast<uint32_t>(__popc(gtm)) << 16) | __popc(cm), S.wsh[1]);
    const uint32_t tot = sc.y;
    uint32_t o = sc.x & 0xFFFFu;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
      if ((cm >> i) & 1u) {
        if (o < kClCap) S.cl[o] = u[i];
        ++o;
      }
    // the list padded to a multiple of four keys (read back 16 bytes at a time) with
    // keys outside digit b1, which every later pass skips
    if (tid < 3) {
      const uint32_t n_here = tot & 0xFFFFu, pad = n_here + static_cast<uint32_t>(tid);
      if ((pad & ~3u) == (n_here & ~3u) && (n_here & 3u) != 0 && pad < static_cast<uint32_t>(kClCap))
        S.cl[pad] = static_cast<uint32_t>(b1 ^ 1) << 21;
    }
    // every CTA of the cluster has started (and zeroed) before any writes into it
    if (pending) {
      cluster_wait();
      pending = false;
    }
    if (tid < static_cast<int>(csize)) {
      st_cluster_u32(cluster_map(smem_u32(&S.meta[rank]), tid), tot);
      st_cluster_u32(cluster_map(smem_u32(&S.meta_b1[rank]), tid), static_cast<uint32_t>(b1));
    }
    if (multi) cluster_sync();
    else __syncthreads();
    if (PRE && round == 0 && rank == 0) gh[tid] = make_uint4(0u, 0u, 0u, 0u);   // every CTA has read it
    G = 0;
    Cc = 0;
    bool agree = true;
    for (uint32_t r = 0; r < csize; ++r) {
      G += S.meta[r] >> 16;
      Cc += S.meta[r] & 0xFFFFu;
      agree = agree && S.meta_b1[r] == static_cast<uint32_t>(b1);
    }
    // A hint that is not an exact histogram (a workspace not left zeroed) can make
    // the bin search ambiguous, so the CTAs may have picked different digits: the
    // counts decide only when every CTA used the same one.
    if (!PRE || (agree && G < k && k <= G + Cc)) break;   // uniform over the cluster
    exchange = true;
  }

  // ---- step 3: the threshold key T, the keys equal to T to take (need_eq), and
  // this CTA's share: selections before it (base) and equal keys taken here (take)
  uint32_t T, base, take, excl;   // excl: this thread's (above T) << 16 | (equal to T) before it in the CTA
  const bool gathered = Cc <= static_cast<uint32_t>(kClCap);
  if (gathered) {
    // cum4[r]: 16-byte groups of the padded lists of the CTAs before r (all ones past
    // the cluster); lo4 / hi4: this CTA's groups
    uint32_t cum4[kClMaxCtas];
    uint32_t lo4 = 0, hi4 = 0, G_lo = 0, n4 = 0;
#pragma unroll
    for (int r = 0; r < kClMaxCtas; ++r) {
      cum4[r] = r < static_cast<int>(csize) ? n4 : 0xFFFFFFFFu;
      if (r < static_cast<int>(csize)) {
        const uint32_t m = S.meta[r];
        if (static_cast<uint32_t>(r) < rank) G_lo += m >> 16;
        if (static_cast<uint32_t>(r) == rank) lo4 = n4;
        n4 += ((m & 0xFFFFu) + 3u) >> 2;
        if (static_cast<uint32_t>(r) == rank) hi4 = n4;
      }
    }
    const uint32_t in_b1 = static_cast<uint32_t>(b1);
    uint4 lv[kClPer4];
#pragma unroll
    for (int m = 0; m < kClPer4; ++m) {
      const uint32_t g4 = static_cast<uint32_t>(tid + m * kClThreads);
      lv[m] = make_uint4(0u, 0u, 0u, 0u);
      if (g4 < n4) {
        uint32_t r = 0, br = 0;
#pragma unroll
        for (int q = 1; q < kClMaxCtas; ++q)
          if (g4 >= cum4[q]) {
            r = static_cast<uint32_t>(q);
            br = cum4[q];
          }
        lv[m] = ld_cluster_v4(cluster_map(smem_u32(&S.cl[4 * (g4 - br)]), r));
      }
    }
#pragma unroll
    for (int m = 0; m < kClPer4; ++m) {
      const uint32_t kv[4] = {lv[m].x, lv[m].y, lv[m].z, lv[m].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (static_cast<uint32_t>(tid + m * kClThreads) < n4 && (kv[e] >> 21) == in_b1)
          atomicAdd(&S.h2[(kv[e] >> 10) & 2047u], 1u);
    }
    __syncthreads();
    // done with the other CTAs' shared memory (their loads consumed above; the wait is before the exit)
    if (multi) cluster_arrive_relaxed();
    const uint2 fA = cl_find(*reinterpret_cast<const uint4*>(&S.h2[4 * tid]), k - G, S.wsh[2], S.res);
    const uint32_t bA = fA.x, a2 = fA.y;
    const uint32_t pre2 = (in_b1 << 11) | bA;
#pragma unroll
    for (int m = 0; m < kClPer4; ++m) {
      const uint32_t kv[4] = {lv[m].x, lv[m].y, lv[m].z, lv[m].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (static_cast<uint32_t>(tid + m * kClThreads) < n4 && (kv[e] >> 10) == pre2) atomicAdd(&S.h3[kv[e] & 1023u], 1u);
    }
    __syncthreads();
    const uint2 fB = cl_find(tid < 256 ? *reinterpret_cast<const uint4*>(&S.h3[4 * tid]) : make_uint4(0u, 0u, 0u, 0u),
                             k - G - a2, S.wsh[3], S.res);
    const uint32_t a3 = fB.y;
    T = (in_b1 << 21) | (bA << 10) | fB.x;
    const uint32_t need_eq = k - G - a2 - a3;
    uint32_t x = 0, y = 0;   // candidates of earlier CTAs above | equal to T; this CTA's equal to T
#pragma unroll
    for (int m = 0; m < kClPer4; ++m) {
      const uint32_t g4 = static_cast<uint32_t>(tid + m * kClThreads);
      const uint32_t kv[4] = {lv[m].x, lv[m].y, lv[m].z, lv[m].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((kv[e] >> 21) != in_b1) continue;   // padding
        if (g4 < lo4) x += (static_cast<uint32_t>(kv[e] > T) << 16) | static_cast<uint32_t>(kv[e] == T);
        else if (g4 < hi4) y += kv[e] == T;
      }
    }
    // this CTA's keys above / equal to T, scanned in position order, together with
    // the sums of x and y (one barrier)
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      gt += i < nv && u[i] > T;
      eq += i < nv && u[i] == T;
    }
    excl = cl_scan_sum2((gt << 16) | eq, x, y, S.wsh[4], S.wsh[5]);
    const uint32_t eq_lo = min(x & 0xFFFFu, need_eq);
    base = G_lo + (x >> 16) + eq_lo;
    take = min(y, need_eq - eq_lo);
  } else {
    // digits 2 and 3 through the cluster (owned bins in hr2 / hr3)
    uint32_t pmask = 0xFFE00000u, pval = static_cast<uint32_t>(b1) << 21, kk = k - G;
#pragma unroll 1
    for (int d = 1; d < 3; ++d) {
      const int shift = d == 1 ? 10 : 0;
      const uint32_t nb = d == 1 ? 2048u : 1024u;
      uint32_t* h = d == 1 ? S.h2 : S.h3;
      uint32_t* hrr = d == 1 ? S.hr2 : S.hr3;
#pragma unroll
      for (int i = 0; i < kPerThread; ++i)
        if (i < nv && (u[i] & pmask) == pval) atomicAdd(&h[(u[i] >> shift) & (nb - 1)], 1u);
      __syncthreads();
      uint4 cc = make_uint4(0u, 0u, 0u, 0u);
      const uint32_t b0 = 4u * tid;
      if (multi) {
        const uint32_t own = ((nb + csize - 1) / csize + 3u) & ~3u;
        for (uint32_t b = tid; b < nb; b += kClThreads) {
          const uint32_t v = h[b];
          if (v == 0) continue;
          const uint32_t o = b / own;
          red_cluster_add(cluster_map(smem_u32(&hrr[b - o * own]), o), v);
        }
        cluster_sync();
        if (b0 < nb) {
          const uint32_t o = b0 / own;
          cc = ld_cluster_v4(cluster_map(smem_u32(&hrr[b0 - o * own]), o));
        }
      } else if (b0 < nb) {
        cc = *reinterpret_cast<const uint4*>(&h[b0]);
      }
      const uint2 f = cl_find(cc, kk, S.wsh[1 + d], S.res);
      pval |= f.x << shift;
      pmask |= (nb - 1) << shift;
      kk -= f.y;
    }
    T = pval;
    const uint32_t need_eq = kk;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      gt += i < nv && u[i] > T;
      eq += i < nv && u[i] == T;
    }
    const uint2 sc = cl_excl_scan((gt << 16) | eq, S.wsh[4]);
    const uint32_t tot = sc.y;
    excl = sc.x;
    if (tid < static_cast<int>(csize)) st_cluster_u32(cluster_map(smem_u32(&S.counts[rank]), tid), tot);
    if (multi) cluster_sync();   // the last access to another CTA's shared memory is before this
    else __syncthreads();
    uint32_t eq_before = 0;
    base = 0;
    for (uint32_t r = 0; r < rank; ++r) {
      const uint32_t cr = S.counts[r];
      const uint32_t e = cr & 0xFFFFu;
      const uint32_t left = need_eq > eq_before ? need_eq - eq_before : 0u;
      base += (cr >> 16) + min(e, left);
      eq_before += e;
    }
    take = min(tot & 0xFFFFu, need_eq > eq_before ? need_eq - eq_before : 0u);
  }

  // ---- step 4: this CTA's selections in position order
  uint32_t eq_rank = excl & 0xFFFFu;
  uint32_t o = base + (excl >> 16) + min(eq_rank, take);
  uint32_t flags = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    bool sel = i < nv && u[i] > T;
    if (i < nv && u[i] == T) sel = eq_rank++ < take;
    flags |= static_cast<uint32_t>(sel) << i;
  }
  while (flags) {
    const int s = s0 + __ffs(flags) - 1;
    flags &= flags - 1;
    if (o < k) {   // exactly k are selected; the guard only bounds the stores
      out[o] = s;
      if (phys) phys[o] = one_block ? ((blk << p.log2_bs) | (s & bs_mask)) : emit_phys(p, btrow, s, bs_mask);
    }
    ++o;
  }
  if (gathered && multi) cluster_wait();   // no CTA leaves while another may still read its candidates
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t st, bool chained, bool zeroed) {
  if (p.b.T == 0) return cudaSuccess;
  if (p.b.max_ctx <= kClMaxRow) {
    const unsigned csize = static_cast<unsigned>(cdiv(p.b.max_ctx, kClSlice));
    if (p.pre_hist)
      return launch_ex(topk_cluster_kernel<true>, dim3(csize, p.b.T), dim3(kClThreads), 0, st, chained, csize, p);
    return launch_ex(topk_cluster_kernel<false>, dim3(csize, p.b.T), dim3(kClThreads), 0, st, chained, csize, p);
  }
  const dim3 grid(p.nchunks, p.b.T);
  cudaError_t e = cudaSuccess;
  if (!zeroed && (e = cudaMemsetAsync(p.zero_begin, 0, p.zero_bytes, st)) != cudaSuccess) return e;
  // each pass starts while the one before drains (programmatic launch; each waits
  // for the one before before it reads anything that one writes)
  if ((e = launch_ex(topk_hist_kernel, grid, dim3(kTopkThreads), 0, st, chained && zeroed, 0u, p)) != cudaSuccess)
    return e;
  if ((e = launch_ex(topk_candidates_kernel, grid, dim3(kTopkThreads), 0, st, true, 0u, p)) != cudaSuccess) return e;
  if ((e = launch_ex(topk_resolve_kernel, dim3(p.b.T), dim3(kResolveThreads), 0, st, true, 0u, p)) != cudaSuccess)
    return e;
  return launch_ex(topk_emit_kernel, grid, dim3(kTopkThreads), 0, st, true, 0u, p);
}

}  // namespace dsa

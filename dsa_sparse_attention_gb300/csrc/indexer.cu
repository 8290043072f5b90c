// indexer.cu — lightning-indexer scoring on the 5th-generation tensor cores.
//
// vLLM K3.1 Pro day-0 post, "Sparse Attention in K3.1 Pro": every earlier token
// is scored for each query with 32 light heads against one FP8 index key,
//   score(t, s) = sum_h w[t,h] * ReLU(q_idx[t,h,:] . key(s)),  key(s) = code(s) * scale(s).
// "Low-latency decode: a fused DSA decode path" describes the scorer as
// key-balanced; "AMD / Quantization" notes keys are reused across query rows
// during speculative verification.  Both hold here:
//  * The contraction is a dense GEMM per 128-key tile: D[key, (token,head)] =
//    keys[128 x 128 B e4m3] x q_idx^T, M = 128 keys, N = 32 heads x (tokens of
//    the group, 1..8), K = 128, tcgen05.mma kind::f8f6f4 with fp32 accumulation
//    in TMEM.  A group's tokens share every key tile (one HBM read per key).
//  * The grid is persistent; each CTA takes an equal contiguous range of the
//    global key-tile enumeration (key-balanced across requests and groups).
//  * Warp roles: producer warps take tiles in turn and stream key pages with TMA
//    (3-D map over the packed pool: 128 B x block slots x rows, 128-byte swizzle,
//    L2 evict-first) plus the per-token scales with bulk copies; producer 0 also
//    loads each group's queries; two MMA warps take tiles in turn; warps 2..9,
//    two sets of four taking alternate tiles, read the accumulators (thread = key)
//    and reduce sum_h w * ReLU(acc) * scale into fp32 scores.  FP8 keys: producers
//    0 and 10..12, MMA warps 1 and 13.  MXFP4 keys: the tensor copy widens each
//    16 packed e2m1 codes to a 16-byte unit (8 bytes of codes, 8 of padding), the
//    operand layout of the block-scaled kind::mxf8f6f4 MMA with E2M1 keys; scale
//    warps 10..13 move each tile's E8M0 exponents into TMEM, where the MMA
//    applies them per 32-dim block; producers 0 and 14..16, MMA warps 1 and 17.
// Page translation (row = block_table[req][s / bs]) happens in the producer.
// Inside a layer step (one token per group) the epilogue also counts each
// token's scores by the top 11 bits of their order-preserving key, the first
// digit of the top-k's radix select, so the top-k starts from that histogram.
#include <cuda.h>

#include "mla_q.cuh"
#include "params.cuh"

namespace dsa {

// ------------------------------------------------------------------ planning

struct PlanParams {
  BatchView b;
  int G;                 // max tokens per group
  ScoreGroup* groups;    // [T], zeroed by the host
  PlanHeader* hdr;
  uint32_t* status;
};

template <typename Op>
__device__ int block_inclusive_scan(int v, int* sh, Op op, int identity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = op(v, x);
  }
  if (lane == 31) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int x = lane < nw ? sh[lane] : identity;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x = op(x, y);
    }
    sh[lane] = x;
  }
  __syncthreads();
  if (warp > 0) v = op(v, sh[warp - 1]);
  __syncthreads();
  return v;
}

struct OpAdd { __device__ int operator()(int a, int b) const { return a + b; } };
struct OpMax { __device__ int operator()(int a, int b) const { return a > b ? a : b; } };

// Splits the tokens into groups: maximal runs of consecutive tokens of the same
// request, cut into pieces of at most G; then counts each group's key tiles.
__global__ void __launch_bounds__(1024) plan_groups_kernel(PlanParams p) {
  __shared__ int sh[32];
  __shared__ int carry_run, carry_groups;
  if (threadIdx.x == 0) { carry_run = 0; carry_groups = 0; }
  __syncthreads();
  const int T = p.b.T;
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    const bool valid = t < T;
    int req = 0, pos = 0, prev = -1;
    if (valid) {
      load_token(p.b, t, p.status, req, pos);
      if (t > 0) {
        int pr = p.b.q_req[t - 1];
        prev = (pr < 0 || pr >= p.b.B) ? (pr < 0 ? 0 : p.b.B - 1) : pr;
      }
    }
    const int rs = (valid && (t == 0 || req != prev)) ? t : -1;
    int run_start = block_inclusive_scan(rs, sh, OpMax(), -1);
    run_start = run_start > carry_run ? run_start : carry_run;
    const int is_start = (valid && ((t - run_start) % p.G == 0)) ? 1 : 0;
    const int incl = block_inclusive_scan(is_start, sh, OpAdd(), 0);
    const int g = carry_groups + incl - 1;
    if (valid) {
      if (is_start) { p.groups[g].t0 = t; p.groups[g].req = req; }
      atomicAdd(&p.groups[g].n, 1);
      atomicMax(&p.groups[g].L, pos + 1);
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      carry_run = run_start;
      carry_groups += incl;
    }
    __syncthreads();
  }
  __syncthreads();
  const int ng = carry_groups;
  __shared__ int chunk_total;
  int carry_tiles = 0;
  for (int base = 0; base < ng; base += blockDim.x) {
    const int g = base + threadIdx.x;
    const int tiles = g < ng ? static_cast<int>(cdiv(__ldcg(&p.groups[g].L), kKeyTile)) : 0;
    const int incl = block_inclusive_scan(tiles, sh, OpAdd(), 0);
    if (g < ng) p.groups[g].tile_begin = carry_tiles + incl - tiles;
    if (threadIdx.x == blockDim.x - 1) chunk_total = incl;
    __syncthreads();
    carry_tiles += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.hdr->n_groups = ng;
    p.hdr->total_tiles = carry_tiles;
  }
}

// ------------------------------------------------------------------- scorer


constexpr int kRowBatch = 32;      // tiles whose block-table rows a producer warp resolves at once (one per lane)
constexpr int kHistBins = 2048;    // top-digit bins of the score histogram handed to the top-k

// Shared-memory / TMEM plan of the scorer.  IDXF = DSA_IDX_FP8 (0) or
// DSA_IDX_MXFP4 (1); G = max tokens per group (N = 32 G).  MXFP4 keys (64 B of
// codes per key in the pool) land as 128 B per key, each 8 bytes of codes padded
// to 16; scale warps move each key's four E8M0 exponents into TMEM, where the
// block-scaled MMA applies exponent b to the products of dims 32b..32b+31 (exact
// powers of two), so one accumulator holds the scaled score terms.
template <int IDXF, int G>
struct ScorerCfg {
  static constexpr bool MX = IDXF == 1;
  // Key stages are freed as soon as their MMA completes; the per-key scales the
  // epilogue reads live in a separate, longer ring of SSLOTS slots.
  static constexpr int STAGES = 8;
  static constexpr int SSLOTS = STAGES + 4;
  static constexpr int ACC_COLS = 32 * G;
  static constexpr int NACC = G == 1 ? 4 : 2;               // TMEM accumulators (even: set = tile parity)
  // MMA issue costs the issuing thread a few hundred cycles per tile, so NMMA
  // warps take tiles in turn (each with its own accumulators).
  static constexpr int NMMA = 2;
  // MXFP4: the block scales of the MMA, A (keys) 4 columns per key stage (key r of
  // the stage at lane r, column r / 32), B (the queries: all 2^0, or with MXFP4
  // queries their exponents) SFB_STRIDE columns per query buffer (token j at column
  // j).  A scale address at an odd column (161) faulted with a misaligned address
  // where columns 160 and 162 worked; every scale region here starts at a multiple
  // of 4.
  static constexpr int SFA_COL = NACC * ACC_COLS;
  static constexpr int SFB_COL = SFA_COL + 4 * STAGES;
  static constexpr int SFB_STRIDE = (G + 3) / 4 * 4;
  static constexpr int TMEM_USED = MX ? SFB_COL + 2 * SFB_STRIDE : NACC * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                   : TMEM_USED <= 64  ? 64
                                   : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256
                                                      : 512;   // allocations are powers of two
  // 16 KB of MMA operand per stage: e4m3 codes, or e2m1 codes with every 8 bytes padded to 16
  static constexpr int KEY_BYTES = kKeyTile * kIdxDim;
  static constexpr int SCALE_BYTES = kKeyTile * 4;
  static constexpr int Q_BYTES = G * kIdxHeads * kIdxDim;
  static constexpr int W_BYTES = G * kIdxHeads * 4;
  static constexpr int OFF_Q = STAGES * KEY_BYTES;
  static constexpr int OFF_QS = OFF_Q + 2 * Q_BYTES;              // MXFP4 queries: 2 x [G][32] E8M0 words
  static constexpr int OFF_SCALES = OFF_QS + (MX ? 2 * G * kIdxHeads * 4 : 0);
  static constexpr int OFF_W = OFF_SCALES + SSLOTS * SCALE_BYTES;   // 2 x [G][32] fp32
  static constexpr int OFF_POS = OFF_W + 2 * W_BYTES;                // 2 x [G] int
  static constexpr int OFF_BARS = OFF_POS + 2 * G * 4 + 64;
  static constexpr int N_BARS = 3 * STAGES + 2 * NACC + 4 + NMMA + 2 * SSLOTS + 2;
  static constexpr int OFF_MISC = OFF_BARS + N_BARS * 8;
  static constexpr int OFF_PLAN = OFF_MISC + 64;            // direct mode: groups [kDirectMaxT] + total
  // Copies are issued by NPROD producer warps taking tiles in turn: one thread
  // issues a bulk or tensor copy in about 150 cycles, several warps in parallel
  // several times faster.
  static constexpr int NPROD = 4;
  static constexpr int OFF_ROWS = OFF_PLAN + kDirectMaxT * 32 + 64;   // producers: [NPROD][kRowBatch][8] block ids
  // One token per group: the epilogue counts the top 11 key bits of its first
  // token's scores in shared memory (later tokens go straight to global memory).
  static constexpr bool HIST = G == 1;
  static constexpr int OFF_HIST = (OFF_ROWS + NPROD * kRowBatch * 8 * 4 + 15) & ~15;   // zeroed 16 bytes at a time
  static constexpr int SMEM_BYTES = OFF_HIST + (HIST ? kHistBins * 4 : 0) + 1024;  // + slack for alignment
  static constexpr int SCALE_WARPS = MX ? 4 : 0;           // one per TMEM lane quarter
  static constexpr int PROD_WARP0 = 10 + SCALE_WARPS;     // producer warps: 0 and PROD_WARP0 ..
  static constexpr int MMA_WARP1 = PROD_WARP0 + NPROD - 1;   // MMA warps: 1 and MMA_WARP1 ..
  static constexpr int THREADS = 320 + 32 * SCALE_WARPS + 32 * (NPROD - 1) + 32 * (NMMA - 1);
  static_assert(NACC % NMMA == 0, "accumulators per MMA warp");
  // Tile i uses stage i % STAGES, producer i % NPROD, MMA warp i % NMMA and scale
  // slot i % SSLOTS.  Each ring's length is a multiple of the number of warps
  // taking tiles in turn, so every slot has one producer and one consumer warp and
  // their parity waits never run two phases apart.
  static_assert(STAGES % NPROD == 0 && STAGES % NMMA == 0, "key stages per producer and MMA warp");
  static_assert(SSLOTS % NPROD == 0 && SSLOTS % 2 == 0, "scale slots per producer and epilogue set");
  static_assert(NACC % 2 == 0, "accumulators per epilogue set");
  static_assert(TMEM_USED <= 512, "tmem columns");
  static_assert(SFA_COL % 4 == 0 && SFB_COL % 4 == 0 && SFB_STRIDE % 4 == 0, "scale addresses at multiples of 4");
  static_assert(SMEM_BYTES <= 232448, "smem");
  static_assert(OFF_HIST % 16 == 0 && OFF_Q % 1024 == 0 && OFF_SCALES % 16 == 0 && OFF_W % 16 == 0 && OFF_BARS % 8 == 0,
                "alignment of the shared-memory regions");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ int find_group(const ScoreGroup* groups, int ng, int tile) {
  int lo = 0, hi = ng - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (groups[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Walks a CTA's tile range, tracking the group each tile belongs to.
struct GroupCursor {
  const ScoreGroup* groups;
  int ng, total, g, next_begin, count;
  ScoreGroup grp;
  __device__ void init(const ScoreGroup* gs, int n, int tot, int tile) {
    groups = gs;
    ng = n;
    total = tot;
    g = find_group(gs, n, tile);
    grp = gs[g];
    next_begin = g + 1 < n ? gs[g + 1].tile_begin : tot;
    count = 0;
  }
  // advance to tile i (called for consecutive i); returns true on a group change
  __device__ bool advance(int i) {
    if (i != next_begin) return false;
    ++g;
    grp = groups[g];
    next_begin = g + 1 < ng ? groups[g + 1].tile_begin : total;
    ++count;
    return true;
  }
};

template <int IDXF, int G>
__global__ void __launch_bounds__(ScorerCfg<IDXF, G>::THREADS, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                   IndexerParams p) {
  using C = ScorerCfg<IDXF, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + C::NACC;
  uint64_t* qfull = tempty + C::NACC;
  uint64_t* qempty = qfull + 2;
  uint64_t* drain = qempty + 2;               // [NMMA]
  uint64_t* sready = drain + C::NMMA;         // [STAGES] MXFP4: the stage's key exponents are in TMEM
  uint64_t* sfull = sready + C::STAGES;       // [SSLOTS] scales landed
  uint64_t* sempty = sfull + C::SSLOTS;       // [SSLOTS] scales read by the epilogue
  uint64_t* qsready = sempty + C::SSLOTS;     // [2] MXFP4 queries: the group's exponents are in TMEM
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  int* abortf = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
  float* wsm = reinterpret_cast<float*>(smem + C::OFF_W);
  int* possm = reinterpret_cast<int*>(smem + C::OFF_POS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);   // the MMA's commit
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], C::NMMA + 8);   // every MMA warp's commit, every epilogue warp
    }
    for (int m = 0; m < C::NMMA; ++m) mbar_init(&drain[m], 1);
    for (int s = 0; s < C::STAGES; ++s) mbar_init(&sready[s], C::SCALE_WARPS > 0 ? C::SCALE_WARPS : 1);
    for (int s = 0; s < C::SSLOTS; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 4);   // the epilogue warps of the tile's set
    }
    for (int i = 0; i < 2; ++i) mbar_init(&qsready[i], C::SCALE_WARPS > 0 ? C::SCALE_WARPS : 1);
    *abortf = 0;
    fence_mbar_init();
    // the descriptors are launch parameters: fetched while the kernel before drains
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&qmap);
  }
  if (warp == 1) tmem_alloc(tslot, C::TMEM_COLS);
  // Everything above touches only this CTA; the inputs may come from the kernel before.
  grid_dep_wait();
  grid_dep_launch();   // a chained top-k may be scheduled as this grid's CTAs retire

  // Plan: groups of tokens and their key-tile ranges.  In direct mode every token
  // is its own group and warp 0 builds the plan here from q_req / q_pos (one global
  // round trip, a warp scan, no block barrier of its own); otherwise
  // plan_groups_kernel wrote it to the workspace.
  ScoreGroup* sg = reinterpret_cast<ScoreGroup*>(smem + C::OFF_PLAN);
  int* plan_total = reinterpret_cast<int*>(smem + C::OFF_PLAN + kDirectMaxT * 32);
  if (p.direct && warp == 0) {
    constexpr int PER = kDirectMaxT / 32;
    const int T = p.b.T;
    int rq[PER], ps[PER];
#pragma unroll
    for (int m = 0; m < PER; ++m) {   // every load issued before any is used
      const int t = lane + 32 * m;
      rq[m] = t < T ? __ldg(p.b.q_req + t) : 0;
      ps[m] = t < T ? __ldg(p.b.q_pos + t) : 0;
    }
    int carry = 0;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      if (32 * m >= T) break;   // uniform: only the warps' worth of tokens present
      const int t = lane + 32 * m;
      int r = rq[m], pos = ps[m], tiles = 0;
      if (t < T) {
        bool bad = false;
        if (r < 0 || r >= p.b.B) { bad = true; r = r < 0 ? 0 : p.b.B - 1; }
        if (pos < 0 || pos >= p.b.max_ctx) { bad = true; pos = pos < 0 ? 0 : p.b.max_ctx - 1; }
        if (bad) atomicOr(p.status, DEV_BAD_BATCH);
        tiles = static_cast<int>(cdiv(pos + 1, kKeyTile));
      }
      int x = tiles;   // inclusive scan over the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (t < T) {
        ScoreGroup g;
        g.t0 = t;
        g.n = 1;
        g.req = r;
        g.L = pos + 1;
        g.tile_begin = carry + x - tiles;
        sg[t] = g;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) *plan_total = carry;
  }
  uint32_t* hs = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);
  const bool hist_on = C::HIST && p.row_hist != nullptr;
  if (hist_on)
    for (int i = threadIdx.x; i < kHistBins / 4; i += C::THREADS) reinterpret_cast<uint4*>(hs)[i] = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();   // the plan, the histogram zeroing and the TMEM address are visible
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const ScoreGroup* groups = p.direct ? sg : p.groups;
  const int total = p.direct ? *plan_total : p.hdr->total_tiles;
  const int ng = p.direct ? p.b.T : p.hdr->n_groups;
  // this CTA's contiguous range of the global tile enumeration (32-bit products when they fit)
  int tile_lo, tile_hi;
  if (static_cast<uint64_t>(total) * gridDim.x < (1ull << 32)) {
    tile_lo = static_cast<int>(blockIdx.x * static_cast<uint32_t>(total) / gridDim.x);
    tile_hi = static_cast<int>((blockIdx.x + 1) * static_cast<uint32_t>(total) / gridDim.x);
  } else {
    tile_lo = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total / gridDim.x);
    tile_hi = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x);
  }
  const Abort ab{abortf, p.status};
  // Layer step with FP8 latents: the epilogue warps, idle until their first tile
  // lands, also write the attention's query terms (one head per warp in turn).
  if (p.mla_q && warp >= 2 && warp < 10) {
    const int total = p.b.T * kMlaHeads, stride = static_cast<int>(gridDim.x) * 8;
#pragma unroll 1
    for (int i = static_cast<int>(blockIdx.x) * 8 + (warp - 2); i < total; i += stride) {
      const int t = i / kMlaHeads, h = i - t * kMlaHeads;
      uint8_t* tok = p.mla_q_terms + static_cast<int64_t>(t) * kQTokenBytes;
      q_head_to_terms(p.mla_q + static_cast<int64_t>(t) * kMlaHeads * kLatDim, h, tok,
                      reinterpret_cast<int32_t*>(tok + kQTermBytes));
    }
  }
  const int bs = p.pool.bs;
  const int box = bs < kKeyTile ? bs : kKeyTile;   // keys per TMA box
  const int nbox = kKeyTile / box;

  if (tile_lo < tile_hi) {
    if (warp == 0 || (warp >= C::PROD_WARP0 && warp < C::MMA_WARP1)) {
      // ------------------------------------------------------------ producers
      // Producer pid takes tiles tile_lo + pid + NPROD m.  Its warp resolves the
      // block-table rows of a batch of its tiles (every load of a lane issued
      // before any is used); lane 0 walks the group cursor over all tiles and
      // issues its tiles' copies.
      const int pid = warp == 0 ? 0 : 1 + warp - C::PROD_WARP0;
      const uint64_t stream_pol = l2_evict_first_policy();
      GroupCursor cur;
      cur.init(groups, ng, total, tile_lo);
      // Producer 0 alone loads the queries, in group order, each group's before
      // the first tile of it that another producer may issue; its waits for a
      // free query buffer therefore never run two phases apart.  A group's
      // buffer is reused two groups later (released by the MMA warps' commits and
      // the epilogue warps).
      GroupCursor qc;
      qc.init(groups, ng, total, tile_lo);
      int q_loaded = 0;                                              // groups whose queries are requested
      auto load_q = [&](const ScoreGroup& grp, int count) -> bool {
        const int qb = count & 1;
        if (count >= 2 && !mbar_wait(&qempty[qb], ((count - 2) >> 1) & 1, ab)) return false;
        for (int j = 0; j < grp.n; ++j) {
          int req, pos;
          if (p.direct) {
            pos = grp.L - 1;
          } else {
            load_token(p.b, grp.t0 + j, p.status, req, pos);
          }
          possm[qb * G + j] = pos;
        }
        // codes (MXFP4: the 4-bit copy counts 64 packed bytes per head), head weights,
        // and with MXFP4 queries their exponents
        const uint32_t code_bytes = C::MX && p.qmx ? kIdxHeads * kIdxDim / 2 : kIdxHeads * kIdxDim;
        const uint32_t qs_bytes = C::MX && p.qmx ? kIdxHeads * 4 : 0;
        mbar_arrive_expect_tx(&qfull[qb], static_cast<uint32_t>(grp.n) * (code_bytes + kIdxHeads * 4 + qs_bytes));
        for (int j = 0; j < grp.n; ++j)
          tma_load_2d(smem + C::OFF_Q + qb * C::Q_BYTES + j * kIdxHeads * kIdxDim, &qmap, &qfull[qb], 0,
                      (grp.t0 + j) * kIdxHeads);
        bulk_load(wsm + qb * G * kIdxHeads, p.w + static_cast<int64_t>(grp.t0) * kIdxHeads,
                  static_cast<uint32_t>(grp.n) * kIdxHeads * 4, &qfull[qb]);
        if (qs_bytes)
          bulk_load(smem + C::OFF_QS + qb * G * kIdxHeads * 4, p.q_scales + static_cast<int64_t>(grp.t0) * kIdxHeads * 4,
                    static_cast<uint32_t>(grp.n) * qs_bytes, &qfull[qb]);
        return true;
      };
      int walked = tile_lo;                                          // tile the cursor is at
      int issued = 0;                                                // this producer's tiles issued
      bool ok = true;
      int* rows_sm = reinterpret_cast<int*>(smem + C::OFF_ROWS) + pid * kRowBatch * 8;   // [kRowBatch][8]
      const int n_mine = tile_hi - tile_lo > pid ? (tile_hi - tile_lo - pid + C::NPROD - 1) / C::NPROD : 0;
      int gb = cur.g;                                                // group of the batch's first tile
      for (int mb = 0; mb < n_mine && ok; mb += kRowBatch) {
        const int nb = min(kRowBatch, n_mine - mb);
        for (int jj = lane; jj < kRowBatch; jj += 32) {
          const int i = tile_lo + pid + (mb + jj) * C::NPROD;
          int idx[kKeyTile / 16];
          int vals[kKeyTile / 16];
          const int32_t* btrow = p.b.bt;
          int L = 0;
          int64_t key0 = 0;
          int g = gb;
          if (jj < nb) {
            while (g + 1 < ng && groups[g + 1].tile_begin <= i) ++g;   // groups span many tiles
            const ScoreGroup gg = groups[g];
            key0 = static_cast<int64_t>(i - gg.tile_begin) * kKeyTile;
            btrow = p.b.bt + static_cast<int64_t>(gg.req) * p.b.bt_stride;
            L = gg.L;
          }
#pragma unroll
          for (int bx = 0; bx < kKeyTile / 16; ++bx) {
            const int64_t k0 = key0 + static_cast<int64_t>(bx) * box;
            idx[bx] = (jj < nb && bx < nbox && k0 < L) ? static_cast<int>(k0 >> p.pool.log2_bs) : -1;
          }
#pragma unroll
          for (int bx = 0; bx < kKeyTile / 16; ++bx) vals[bx] = idx[bx] >= 0 ? __ldg(btrow + idx[bx]) : -1;
#pragma unroll
          for (int bx = 0; bx < kKeyTile / 16; ++bx) {
            int row = vals[bx];
            if (idx[bx] >= 0 && (row < 0 || row >= p.pool.num_rows)) {
              atomicOr(p.status, DEV_BAD_BLOCK);
              row = -1;
            }
            rows_sm[jj * 8 + bx] = idx[bx] >= 0 ? row : -1;
          }
          gb = max(gb, g);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gb = max(gb, __shfl_xor_sync(0xffffffffu, gb, o));
        __syncwarp();
        if (lane == 0) {
          for (int jj = 0; jj < nb; ++jj) {
            const int i = tile_lo + pid + (mb + jj) * C::NPROD;
            while (walked < i) cur.advance(++walked);
            const ScoreGroup& grp = cur.grp;
            if (pid == 0 && q_loaded == 0) {
              if (!(ok = load_q(qc.grp, 0))) break;
              q_loaded = 1;
            }
            const int it = i - tile_lo;
            const int s = it % C::STAGES;
            const int ss = it % C::SSLOTS;
            if (it >= C::STAGES && !(ok = mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1, ab))) break;
            if (it >= C::SSLOTS && !(ok = mbar_wait(&sempty[ss], ((it / C::SSLOTS) - 1) & 1, ab))) break;
            const int* rows = rows_sm + jj * 8;
            const int64_t key0 = static_cast<int64_t>(i - grp.tile_begin) * kKeyTile;
            constexpr int VB = C::MX ? kIdxDim / 2 : kIdxDim;   // value bytes per key in the page (counted)
            uint32_t nkeys = 0;
            for (int bx = 0; bx < nbox; ++bx)
              if (rows[bx] >= 0) nkeys += static_cast<uint32_t>(box);
            mbar_arrive_expect_tx(&full[s], nkeys * VB);
            mbar_arrive_expect_tx(&sfull[ss], nkeys * 4);
            for (int bx = 0; bx < nbox; ++bx) {
              const int row = rows[bx];
              if (row < 0) continue;
              const int64_t k0 = key0 + static_cast<int64_t>(bx) * box;
              const int slot0 = static_cast<int>(k0 & (bs - 1));
              uint8_t* vdst = smem + s * C::KEY_BYTES + bx * box * kIdxDim;   // 128 B per key in shared memory
              tma_load_3d_hint(vdst, &kmap, &full[s], 0, slot0, row, stream_pol);
              const uint8_t* src = p.pool.pool + static_cast<int64_t>(row) * p.pool.row_stride + p.pool.idx_off +
                                   static_cast<int64_t>(bs) * VB + static_cast<int64_t>(slot0) * 4;
              bulk_load_hint(smem + C::OFF_SCALES + ss * C::SCALE_BYTES + bx * box * 4, src, box * 4, &sfull[ss],
                             stream_pol);
            }
            ++issued;
            if (pid == 0) {   // the queries of the groups starting within the next NPROD tiles
              const int ahead = min(i + C::NPROD, tile_hi - 1);
              while (ok && qc.next_begin <= ahead) {
                qc.advance(qc.next_begin);
                if ((ok = load_q(qc.grp, qc.count))) q_loaded = qc.count + 1;
              }
              if (!ok) break;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        __syncwarp();
      }
      if (!ok && lane == 0) {   // drain this producer's copies still in flight before the CTA exits
        for (int m = issued - 1; m >= 0 && m >= issued - C::STAGES; --m) {
          const int it = pid + m * C::NPROD;
          drain_wait(&full[it % C::STAGES], (it / C::STAGES) & 1);
          drain_wait(&sfull[it % C::SSLOTS], (it / C::SSLOTS) & 1);
        }
        for (int c = q_loaded > 2 ? q_loaded - 2 : 0; c < q_loaded; ++c) drain_wait(&qfull[c & 1], (c >> 1) & 1);
      }
    } else if (warp == 1 || warp >= C::MMA_WARP1) {
      // ---------------------------------------------------------- MMA issuers
      // MMA warp mid takes tiles tile_lo + mid + NMMA m; every MMA warp walks the
      // cursor over all tiles and commits the query buffer of each group it passes.
      const int mid = warp == 1 ? 0 : 1 + warp - C::MMA_WARP1;
      if (lane == 0) {
        GroupCursor cur;
        cur.init(groups, ng, total, tile_lo);
        const bool qmx = C::MX && p.qmx;
        auto idesc_of = [qmx](int n) {   // E2M1 keys with e4m3 (or E2M1) queries
          return C::MX ? make_idesc_bs(5, qmx ? 5 : 0, kKeyTile, n * kIdxHeads, 0, 0)
                       : make_idesc(0, 0, false, false, kKeyTile, n * kIdxHeads);
        };
        uint32_t idesc = idesc_of(cur.grp.n);
        bool ok = mbar_wait(&qfull[0], 0, ab) && (!qmx || mbar_wait(&qsready[0], 0, ab));
        for (int i = tile_lo; i < tile_hi && ok; ++i) {
          if (cur.advance(i)) {
            idesc = idesc_of(cur.grp.n);
            if (!(ok = mbar_wait(&qfull[cur.count & 1], (cur.count >> 1) & 1, ab))) break;
            if (qmx && !(ok = mbar_wait(&qsready[cur.count & 1], (cur.count >> 1) & 1, ab))) break;
          }
          const int it = i - tile_lo;
          if (it % C::NMMA == mid) {
            const int s = it % C::STAGES;
            const int acc = it % C::NACC;
            if (!(ok = mbar_wait_inline(&full[s], (it / C::STAGES) & 1, ab))) break;
            if (C::MX && !(ok = mbar_wait_inline(&sready[s], (it / C::STAGES) & 1, ab))) break;
            if (it >= C::NACC && !(ok = mbar_wait_inline(&tempty[acc], ((it / C::NACC) - 1) & 1, ab))) break;
            tc_fence_after();
            const uint32_t d = tmem + acc * C::ACC_COLS;
            const uint32_t a0 = smem_u32(smem + s * C::KEY_BYTES);
            const uint32_t b0 = smem_u32(smem + C::OFF_Q + (cur.count & 1) * C::Q_BYTES);
#pragma unroll
            for (int k = 0; k < kIdxDim / 32; ++k) {
              // one accumulator over K = 128; MXFP4: block k (dims 32k..32k+31) scaled by
              // byte k of each key's exponent cell
              const uint64_t ad = make_sdesc_sw128(a0 + 32 * k, 16, 1024);
              const uint64_t bd = make_sdesc_sw128(b0 + 32 * k, 16, 1024);
              if (C::MX)   // scale byte k: the keys' (and MXFP4 queries') exponent of block k
                mma_mxf8f6f4_bs(d, ad, bd, idesc | (static_cast<uint32_t>(k) << 29) | (qmx ? k << 4 : 0u),
                                tmem + C::SFA_COL + 4 * s, tmem + C::SFB_COL + (cur.count & 1) * C::SFB_STRIDE,
                                k > 0 ? 1u : 0u);
              else
                mma_f8f6f4(d, ad, bd, idesc, k > 0 ? 1u : 0u);
            }
            tc_commit(&empty[s]);
            tc_commit(&tfull[acc]);
          }
          if (i + 1 == cur.next_begin || i + 1 == tile_hi) tc_commit(&qempty[cur.count & 1]);
        }
        if (!ok) {
          tc_commit(&drain[mid]);
          drain_wait(&drain[mid], 0);
        }
      }
    } else if (C::MX && warp >= 10 && warp < C::PROD_WARP0) {
      // ------------------------------------------------- scale warps (MXFP4)
      // The warp of lane quarter q writes the E8M0 cells of keys 32q .. 32q+31 of
      // each tile into TMEM (lane = key, column SFA_COL + 4 s + q: the layout the
      // block-scaled MMA reads) once the stage's previous MMA is done with them,
      // and, before its first tile, the query's unit scales in its quarter.
      const int q = warp & 3;
      const uint32_t lq = static_cast<uint32_t>(32 * q) << 16;
      const bool qmx = p.qmx != 0;
      if (!qmx)
        for (int c = 0; c < 2 * C::SFB_STRIDE; ++c) tmem_st1(tmem + lq + C::SFB_COL + c, 0x7F7F7F7Fu);   // 2^0 in every byte
      // MXFP4 queries: a group's head exponents (head h at lane h of every quarter,
      // token j at column SFB_COL + buffer * SFB_STRIDE + j), once its query has landed
      GroupCursor gc;
      gc.init(groups, ng, total, tile_lo);
      auto group_scales = [&](int count) -> bool {
        const int qb = count & 1;
        if (!mbar_wait(&qfull[qb], (count >> 1) & 1, ab)) return false;
        const uint32_t* qs = reinterpret_cast<const uint32_t*>(smem + C::OFF_QS) + qb * G * kIdxHeads;
        for (int j = 0; j < gc.grp.n; ++j)
          tmem_st1(tmem + lq + C::SFB_COL + qb * C::SFB_STRIDE + j, qs[j * kIdxHeads + lane]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qsready[qb]);
        return true;
      };
      bool ok = !qmx || tile_lo >= tile_hi || group_scales(0);
      for (int i = tile_lo; i < tile_hi && ok; ++i) {
        if (gc.advance(i) && qmx && !(ok = group_scales(gc.count))) break;
        const int it = i - tile_lo;
        const int s = it % C::STAGES, ss = it % C::SSLOTS;
        if (it >= C::STAGES && !(ok = mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1, ab))) break;
        if (!(ok = mbar_wait(&sfull[ss], (it / C::SSLOTS) & 1, ab))) break;
        const uint32_t e8 = reinterpret_cast<const uint32_t*>(smem + C::OFF_SCALES + ss * C::SCALE_BYTES)[32 * q + lane];
        tmem_st1(tmem + lq + C::SFA_COL + 4 * s + q, e8);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sready[s]);
      }
      tmem_wait_st();   // none in flight at the deallocation (also after an abort)
    } else {
      // ------------------------------------------------------------ epilogue
      // Two sets of four warps take alternate tiles; in a set, warp w reads TMEM
      // lanes 32*(w%4).. (one key per thread) and reduces all the group's tokens.
      const int e = warp - 2;
      const int quarter = warp & 3;
      const int set = e >> 2;
      GroupCursor cur;
      cur.init(groups, ng, total, tile_lo);
      const int first_t = cur.grp.t0;
      bool ok = mbar_wait(&qfull[0], 0, ab);
      for (int i = tile_lo; i < tile_hi && ok; ++i) {
        if (cur.advance(i)) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&qempty[(cur.count - 1) & 1]);   // done with the previous group
          if (!(ok = mbar_wait(&qfull[cur.count & 1], (cur.count >> 1) & 1, ab))) break;
        }
        const int it = i - tile_lo;
        if ((it & 1) != set) continue;
        const int ss = it % C::SSLOTS;
        const int acc = it % C::NACC;
        if (!(ok = mbar_wait(&tfull[acc], (it / C::NACC) & 1, ab))) break;
        if (!(ok = mbar_wait(&sfull[ss], (it / C::SSLOTS) & 1, ab))) break;
        tc_fence_after();
        const ScoreGroup& grp = cur.grp;
        const int qb = cur.count & 1;
        const int kloc = quarter * 32 + lane;
        const int key = (i - grp.tile_begin) * kKeyTile + kloc;
        // FP8: the key's fp32 scale; MXFP4: already applied by the MMA
        const float scale = C::MX ? 1.f : reinterpret_cast<const float*>(smem + C::OFF_SCALES + ss * C::SCALE_BYTES)[kloc];
        // one token's 32 head sums -> its score (and the histogram hand-off)
        auto finish = [&](const uint32_t (&r)[32], int j) {
          const float4* wv = reinterpret_cast<const float4*>(wsm + (qb * G + j) * kIdxHeads);
          float sum = 0.f;
          if (scale >= 0.f) {
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
              const float4 w4 = wv[h4];
              sum = fmaf(w4.x, fmaxf(__uint_as_float(r[4 * h4 + 0]), 0.f), sum);
              sum = fmaf(w4.y, fmaxf(__uint_as_float(r[4 * h4 + 1]), 0.f), sum);
              sum = fmaf(w4.z, fmaxf(__uint_as_float(r[4 * h4 + 2]), 0.f), sum);
              sum = fmaf(w4.w, fmaxf(__uint_as_float(r[4 * h4 + 3]), 0.f), sum);
            }
          } else {   // ReLU(c * x) = c * min(x, 0) for c < 0
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
              const float4 w4 = wv[h4];
              sum = fmaf(w4.x, fminf(__uint_as_float(r[4 * h4 + 0]), 0.f), sum);
              sum = fmaf(w4.y, fminf(__uint_as_float(r[4 * h4 + 1]), 0.f), sum);
              sum = fmaf(w4.z, fminf(__uint_as_float(r[4 * h4 + 2]), 0.f), sum);
              sum = fmaf(w4.w, fminf(__uint_as_float(r[4 * h4 + 3]), 0.f), sum);
            }
          }
          const int pos = possm[qb * G + j];
          if (key <= pos) {
            const float v = scale * sum;
            p.scores[static_cast<int64_t>(grp.t0 + j) * p.ld + key] = v;
            if (hist_on) {
              const uint32_t bin = score_key(v) >> 21;
              if (cur.count == 0) atomicAdd(&hs[bin], 1u);
              else atomicAdd(p.row_hist + static_cast<int64_t>(grp.t0 + j) * kHistBins + bin, 1u);
            }
          }
        };
        // groups of several tokens: two tokens' sums per TMEM wait (a wait covers
        // every load before it, so loads issued together share one latency)
        constexpr bool PAIR = !C::MX && G > 1;   // MXFP4 kernels have no registers to spare
        for (int j = 0; j < grp.n; j += PAIR ? 2 : 1) {
          const bool two = PAIR && j + 1 < grp.n;   // warp-uniform
          uint32_t r[32], r2[32];
          DSA_TMEM_LD32(tmem + acc * C::ACC_COLS + j * kIdxHeads + (static_cast<uint32_t>(quarter * 32) << 16), r);
          if (two)
            DSA_TMEM_LD32(tmem + acc * C::ACC_COLS + (j + 1) * kIdxHeads + (static_cast<uint32_t>(quarter * 32) << 16),
                          r2);
          tmem_wait_ld();
          finish(r, j);
          if (two) finish(r2, j + 1);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tempty[acc]);
          mbar_arrive(&sempty[ss]);
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&qempty[cur.count & 1]);
      if (hist_on) {
        // every epilogue warp leaves the loop (finished or aborted) and meets here
        named_bar_sync(1, 256);
        uint32_t* dst = p.row_hist + static_cast<int64_t>(first_t) * kHistBins;
        for (int b = threadIdx.x - 64; b < kHistBins; b += 256) {
          const uint32_t v = hs[b];
          if (v) atomicAdd(dst + b, v);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ----------------------------------------------------------------- launchers

cudaError_t launch_plan_groups(const BatchView& b, int G, ScoreGroup* groups, PlanHeader* hdr, uint32_t* status,
                               cudaStream_t st) {
  PlanParams p{b, G, groups, hdr, status};
  plan_groups_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

template <int IDXF, int G>
static cudaError_t launch_scorer_g(const CUtensorMap& kmap, const CUtensorMap& qmap, const IndexerParams& p,
                                   int grid, cudaStream_t st) {
  using C = ScorerCfg<IDXF, G>;
  cudaError_t e = set_func_attr_once(reinterpret_cast<const void*>(indexer_kernel<IDXF, G>),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // chained: the set-up above the kernel's wait overlaps the end of the kernel before it
  return launch_ex(indexer_kernel<IDXF, G>, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, st, true, 0u, kmap, qmap, p);
}

int indexer_group_size(int idx_fmt, bool one_token_per_request) {
  if (one_token_per_request) return 1;
  return idx_fmt == 1 ? 2 : 8;
}

cudaError_t launch_indexer(const CUtensorMap& kmap, const CUtensorMap& qmap, const IndexerParams& p, int G,
                           int grid, cudaStream_t st) {
  if (p.pool.idx_fmt == 1) {
    if (G == 1) return launch_scorer_g<1, 1>(kmap, qmap, p, grid, st);
    return launch_scorer_g<1, 2>(kmap, qmap, p, grid, st);
  }
  if (G == 1) return launch_scorer_g<0, 1>(kmap, qmap, p, grid, st);
  return launch_scorer_g<0, 8>(kmap, qmap, p, grid, st);
}

}  // namespace dsa

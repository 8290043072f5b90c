// front.cu — the fused indexer front and the new tokens' cache writes.
//
// vLLM K3.1 Pro day-0 post, "Low-latency decode: a fused DSA decode path": one
// kernel applies the query norm, projects the indexer query, quantizes it (FP8 or
// MXFP4) with the head weights absorbing the scales, and writes the new token's
// index key; the new token's latent enters the cache from the MLA query side.
// The post gives no shapes.  Readings: RMSNorm over the compressed query of
// width d_q, q = W . norm(c_q) with W [32 * 128, d_q], FP8 per (token, head) with
// s = max|q_h| / 448 folded into the head weight, the new key FP8 with
// s_k = max|k| / 448, latents FP8 (plain e4m3) or NVFP4 (e4m3 scale max|x| / 6
// per 16 values, e2m1 values).
//
// Indexer front.  At decode the projection is a weight stream (4096 x d_q bf16,
// 12.6 MB at d_q = 1536) against a few queries.  It runs on the tensor cores:
// grid (32 heads x 4 quarters of d_q, token chunks of 8) in clusters of the 4
// quarters of a head.  Each CTA streams its head's 128 rows of W over its quarter
// of d_q into a 6-slot ring by TMA (64 dims, 128-byte swizzle, the K-major A
// operand), while 8 warps normalise the chunk's queries and write them as the B
// operand: per token two bf16 rows, hi = bf16(y) and lo = bf16(y - hi), so that
// W . y is carried to about 2^-17 of each product.  One thread issues
// tcgen05.mma kind::f16 (M = 128 rows, N = 16, fp32 accumulation in TMEM); the
// epilogue adds the hi and lo columns, and after one cluster barrier the first
// CTA adds the four quarters, takes each token's maximum over the head and writes
// the codes and folded weights; the second CTA of the first head meanwhile writes
// the chunk's new index keys.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "../../include/dsa.h"
#include "params.cuh"

namespace dsa {

namespace front {
constexpr int THREADS = 320;             // warps 0..7: queries, 0..3 also the epilogue; 8: W copies; 9: MMA
constexpr int PROD_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int CHUNK = 8;                 // query tokens per CTA
constexpr int ROWS = 32;                 // rows (dims of one head) a CTA finalises
constexpr int MAX_DQ = 4096;
constexpr int KC = 64;                   // dims per W copy and B chunk (one 128-byte row of bf16)
constexpr int RING = 6;                  // W copies in flight
constexpr int MAX_CPQ = (MAX_DQ / KC + 3) / 4;   // chunks of one quarter of d_q
constexpr int A_BYTES = 128 * KC * 2;    // 128 rows of W x 64 dims
constexpr int B_CHUNK = 16 * KC * 2;     // 16 rows (8 tokens, hi | lo) x 64 dims
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + RING * A_BYTES;
constexpr int OFF_RED = OFF_B + MAX_CPQ * B_CHUNK;
constexpr int OFF_QV = OFF_RED + 4 * ROWS * CHUNK * 4;
constexpr int OFF_AMAX = OFF_QV + ROWS * CHUNK * 4;
constexpr int OFF_BARS = OFF_AMAX + 2 * CHUNK * 4;
constexpr int OFF_MISC = OFF_BARS + (2 * RING + 1) * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + alignment slack
static_assert(OFF_B % 1024 == 0 && A_BYTES % 1024 == 0 && B_CHUNK % 1024 == 0, "swizzled operands");
static_assert(OFF_BARS % 8 == 0, "barriers");
}  // namespace front

// Physical row and slot of token t's position (checked); false when out of range.
__device__ __forceinline__ bool new_token_slot(const BatchView& b, const PoolView& pool, int t, uint32_t* status,
                                               int64_t& row, int& slot) {
  int req, pos;
  load_token(b, t, status, req, pos);
  const int64_t blk = pos >> pool.log2_bs;
  if (blk >= b.bt_stride) {
    atomicOr(status, DEV_BAD_BATCH);
    return false;
  }
  row = __ldg(b.bt + static_cast<int64_t>(req) * b.bt_stride + blk);
  if (row < 0 || row >= pool.num_rows) {
    atomicOr(status, DEV_BAD_BLOCK);
    return false;
  }
  slot = pos & (pool.bs - 1);
  return true;
}

__device__ __forceinline__ uint32_t f4_to_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
  const uint32_t hi = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3));
  return lo | (hi << 16);
}

__global__ void __launch_bounds__(front::THREADS, 1)
    indexer_front_kernel(const __grid_constant__ CUtensorMap wmap, FrontParams p) {
  using namespace front;
  extern __shared__ uint8_t fsm_raw[];
  uint8_t* fsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fsm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = fsm + OFF_A;                                        // [RING][128 rows x 128 B] (swizzled)
  uint8_t* bq = fsm + OFF_B;                                          // [MAX_CPQ][16 rows x 128 B] (swizzled)
  float* red = reinterpret_cast<float*>(fsm + OFF_RED);               // [4 quarters][32 rows][8] partial sums
  float* qv = reinterpret_cast<float*>(fsm + OFF_QV);                 // [ROWS][CHUNK] this CTA's rows
  float* amax_sh = reinterpret_cast<float*>(fsm + OFF_AMAX);          // [CHUNK] this CTA's per-token max |q|
  float* amax_all = amax_sh + CHUNK;                                  // [CHUNK] the head's
  uint64_t* bars = reinterpret_cast<uint64_t*>(fsm + OFF_BARS);
  uint64_t* full = bars;                                              // [RING] W chunk landed
  uint64_t* empty = bars + RING;                                      // [RING] its MMAs are done
  uint64_t* done = bars + 2 * RING;                                   // every MMA is done (one phase)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fsm + OFF_MISC);
  int* abortf = reinterpret_cast<int*>(fsm + OFF_MISC + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = static_cast<int>(cluster_rank()), h = blockIdx.x >> 2;
  const int t0 = blockIdx.y * CHUNK;
  const int nt = min(CHUNK, p.b.T - t0);
  const int dq = p.d_q;
  // this CTA's 64-dim chunks of d_q: [c_first, c_first + ncv)
  const int nch = (dq + KC - 1) / KC, cpq = (nch + 3) / 4;
  const int c_first = quarter * cpq;
  const int ncv = max(0, min(cpq, nch - c_first));
  int issued = 0;   // W copies issued (by thread 0 first, then by the producer warp)
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * RING + 1; ++i) mbar_init(&bars[i], 1);
    *abortf = 0;
    fence_mbar_init();
    // The weights are an input of the call that no kernel before writes: their first
    // RING copies start at once (the rest as the MMAs free their slots, below).
    for (; issued < ncv && issued < RING; ++issued) {
      mbar_arrive_expect_tx(&full[issued], A_BYTES);
      tma_load_2d(ring + issued * A_BYTES, &wmap, &full[issued], (c_first + issued) * KC, h * 128);
    }
  }
  if (warp == MMA_WARP) tmem_alloc(tslot, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (warp == PROD_WARP && lane == 0) issued = min(ncv, RING);
  grid_dep_wait();
  const Abort ab{abortf, p.status};
  if (warp < CHUNK) {
    // ---- RMSNorm of token `warp` over all of d_q, then its normalised values in
    // this CTA's dims as two bf16 terms (row warp: hi, row 8 + warp: lo) of the
    // MMA's B operand, K-major with the 128-byte swizzle; zeros past d_q and for
    // absent tokens
    const int t = warp;
    float r = 0.f;
    const __nv_bfloat16* x = p.c_q + static_cast<int64_t>(t0 + t) * dq;
    if (t < nt) {
      float ss = 0.f;
#pragma unroll 1
      for (int i0 = lane * 8; i0 < dq; i0 += 256 * 4) {   // four 16-byte loads in flight per lane
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v[u] = i0 + 256 * u < dq ? __ldg(reinterpret_cast<const uint4*>(x + i0 + 256 * u)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a = __uint_as_float(w4[j] << 16), c = __uint_as_float(w4[j] & 0xFFFF0000u);
            ss = fmaf(a, a, fmaf(c, c, ss));
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      r = 1.0f / sqrtf(ss / static_cast<float>(dq) + p.eps);
    }
    const int k0 = c_first * KC;
    for (int j = lane; j < cpq * (KC / 8); j += 32) {   // 16-byte pieces of the CTA's dims
      const int idx = k0 + 8 * j;
      uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = make_uint4(0u, 0u, 0u, 0u);
      if (t < nt && idx < dq) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + idx));
        const uint4 gm = __ldg(reinterpret_cast<const uint4*>(p.gamma + idx));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w}, g4[4] = {gm.x, gm.y, gm.z, gm.w};
        uint32_t h4[4], l4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float ya = __uint_as_float(w4[e] << 16) * r * __uint_as_float(g4[e] << 16);
          const float yb = __uint_as_float(w4[e] & 0xFFFF0000u) * r * __uint_as_float(g4[e] & 0xFFFF0000u);
          const __nv_bfloat162 hh = __floats2bfloat162_rn(ya, yb);
          const float2 hf = __bfloat1622float2(hh);
          const __nv_bfloat162 ll = __floats2bfloat162_rn(ya - hf.x, yb - hf.y);
          h4[e] = *reinterpret_cast<const uint32_t*>(&hh);
          l4[e] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        hi = make_uint4(h4[0], h4[1], h4[2], h4[3]);
        lo = make_uint4(l4[0], l4[1], l4[2], l4[3]);
      }
      const int c = j / (KC / 8), piece = j % (KC / 8);
      uint8_t* chunk = bq + c * B_CHUNK;
      *reinterpret_cast<uint4*>(chunk + sw128_off(t, piece)) = hi;                 // row t (rows 0..7: atom 0)
      *reinterpret_cast<uint4*>(chunk + 1024 + sw128_off(t, piece)) = lo;          // row 8 + t (atom 1)
    }
    fence_proxy_async_smem();   // visible to the tensor core
  }
  __syncthreads();   // the B operand is complete
  if (warp == PROD_WARP && lane == 0) {
    for (; issued < ncv; ++issued) {
      const int s = issued % RING;
      if (!mbar_wait(&empty[s], ((issued / RING) - 1) & 1, ab)) break;
      mbar_arrive_expect_tx(&full[s], A_BYTES);
      tma_load_2d(ring + s * A_BYTES, &wmap, &full[s], (c_first + issued) * KC, h * 128);
    }
  } else if (warp == MMA_WARP && lane == 0) {
    // ---- D[128 rows][16] (+)= W chunk x B chunk, four K = 16 steps per chunk
    const uint32_t idesc = make_idesc(1, 1, false, false, 128, 16);
    for (int c = 0; c < ncv; ++c) {
      const int s = c % RING;
      if (!mbar_wait(&full[s], (c / RING) & 1, ab)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(ring + s * A_BYTES), b0 = smem_u32(bq + c * B_CHUNK);
#pragma unroll
      for (int k = 0; k < KC / 16; ++k)
        mma_f16(tmem, make_sdesc_sw128(a0 + 32 * k, 16, 1024), make_sdesc_sw128(b0 + 32 * k, 16, 1024), idesc,
                (c > 0 || k > 0) ? 1u : 0u);
      tc_commit(&empty[s]);
    }
    tc_commit(done);   // completes when every MMA issued above has (at once with none)
  }
  __syncwarp();
  // ---- epilogue: warp w < 4 holds rows 32w.. of the head: this quarter's 8 sums per
  // row (hi + lo columns) into its own shared memory; after one cluster barrier the
  // first CTA adds the four quarters, takes the head's maximum per token and writes
  // the codes and the folded weights
  if (warp < 4) {
    float q8[CHUNK];
    const bool ok = mbar_wait(done, 0, ab);
    tc_fence_after();
    if (ok && ncv > 0) {
      uint32_t a[8], b[8];
      DSA_TMEM_LD8(tmem + (static_cast<uint32_t>(warp * 32) << 16), a);
      DSA_TMEM_LD8(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 8, b);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < CHUNK; ++t) q8[t] = __uint_as_float(a[t]) + __uint_as_float(b[t]);
    } else {
#pragma unroll
      for (int t = 0; t < CHUNK; ++t) q8[t] = 0.f;
    }
    float4* dst = reinterpret_cast<float4*>(red + threadIdx.x * CHUNK);   // [128 rows][8]
    dst[0] = make_float4(q8[0], q8[1], q8[2], q8[3]);
    dst[1] = make_float4(q8[4], q8[5], q8[6], q8[7]);
  }
  cluster_arrive();
  cluster_wait();   // every quarter's partial sums are in its shared memory
  if (quarter == 0 && warp < 4) {
    const int row = threadIdx.x;   // dim of head h
    const float hw = row < nt ? __ldg(p.head_w + (t0 + row) * kIdxHeads + h) : 0.f;   // token row's head weight
    float q8[CHUNK];
#pragma unroll
    for (int t = 0; t < CHUNK; ++t) q8[t] = 0.f;
#pragma unroll
    for (uint32_t src = 0; src < 4; ++src) {
      const uint32_t at = cluster_map(smem_u32(red + row * CHUNK), src);
      const uint4 v0 = ld_cluster_v4(at), v1 = ld_cluster_v4(at + 16);
      q8[0] += __uint_as_float(v0.x);
      q8[1] += __uint_as_float(v0.y);
      q8[2] += __uint_as_float(v0.z);
      q8[3] += __uint_as_float(v0.w);
      q8[4] += __uint_as_float(v1.x);
      q8[5] += __uint_as_float(v1.y);
      q8[6] += __uint_as_float(v1.z);
      q8[7] += __uint_as_float(v1.w);
    }
    if (p.qmx) {
      // MXFP4 (uniform over the CTA): warp w holds the head's 32-dim block w of each
      // token, so the block's maximum is a warp maximum.  E = floor(log2 max) - 2 + 127
      // clamped to 0..254 (0 for a zero block), codes e2m1(q * 2^(127 - E)) (an exact
      // power-of-two scaling, then round to nearest even, saturating at 6), two per
      // byte with the even dim in the low nibble; the exponents follow all the codes.
      const int64_t nT = p.b.T;
      uint8_t* cdst = p.q_idx + (static_cast<int64_t>(t0) * kIdxHeads + h) * (kIdxDim / 2) + (row >> 1);
      uint8_t* edst = p.q_idx + nT * kIdxHeads * (kIdxDim / 2) + (static_cast<int64_t>(t0) * kIdxHeads + h) * 4 + warp;
#pragma unroll
      for (int t = 0; t < CHUNK; ++t) {
        float m = fabsf(q8[t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int e = m > 0.f ? min(max(ilogbf(m) - 2 + 127, 0), 254) : 0;
        const float v = q8[t] * __uint_as_float(static_cast<uint32_t>(254 - e) << 23);
        const uint32_t c = __nv_cvt_float_to_fp4(v, __NV_E2M1, cudaRoundNearest) & 0xFu;
        const uint32_t c_odd = __shfl_down_sync(0xffffffffu, c, 1);
        if (t < nt) {
          if ((lane & 1) == 0) cdst[static_cast<int64_t>(t) * kIdxHeads * (kIdxDim / 2)] = static_cast<uint8_t>(c | (c_odd << 4));
          if (lane == 0) edst[static_cast<int64_t>(t) * kIdxHeads * 4] = static_cast<uint8_t>(e);
        }
      }
      if (row < nt) p.w_out[static_cast<int64_t>(t0 + row) * kIdxHeads + h] = hw;   // the scales travel with the codes
    } else {
    // the head's max |q| per token: within the warp, then over the 4 warps
#pragma unroll
    for (int t = 0; t < CHUNK; ++t) {
      float m = fabsf(q8[t]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) qv[warp * CHUNK + t] = m;
    }
    named_bar_sync(1, 128);
    // s = max / 448 (1 for an all-zero head): thread t < 8 takes token t's scale, its
    // reciprocal and its folded weight
    if (row < CHUNK) {
      const float m = fmaxf(fmaxf(qv[row], qv[CHUNK + row]), fmaxf(qv[2 * CHUNK + row], qv[3 * CHUNK + row]));
      const float sc = m > 0.f ? m / 448.0f : 1.0f;
      amax_all[row] = 1.0f / sc;
      if (row < nt) p.w_out[static_cast<int64_t>(t0 + row) * kIdxHeads + h] = hw * sc;
    }
    named_bar_sync(1, 128);
    // codes e4m3(q / s), one byte per token and dim
    uint8_t* qdst = p.q_idx + (static_cast<int64_t>(t0) * kIdxHeads + h) * kIdxDim + row;
#pragma unroll
    for (int t = 0; t < CHUNK; ++t)
      if (t < nt)
        qdst[static_cast<int64_t>(t) * kIdxHeads * kIdxDim] =
            static_cast<uint8_t>(__nv_cvt_float_to_fp8(q8[t] * amax_all[t], __NV_SATFINITE, __NV_E4M3));
    }
  }
  if (quarter != 0) cluster_arrive_relaxed();   // the first CTA reads this one's sums until the end
  // the chunk's new index keys (second quarter of head 0, while the first finalises
  // the head): one warp per token, four values per lane.  FP8 pages: s_k = max |k| /
  // 448 in fp32.  MXFP4 pages: per 32 dims (8 lanes) the MX exponent and e2m1 codes
  // as for the queries, 64 code bytes at the slot, the 4 exponents in the scale area.
  if (p.k_new && blockIdx.x == 1 && warp < nt && p.pool.idx_fmt == DSA_IDX_MXFP4) {
    const int t = t0 + warp;
    const uint2 kv = __ldg(reinterpret_cast<const uint2*>(p.k_new + static_cast<int64_t>(t) * kIdxDim) + lane);
    const float kk[4] = {__uint_as_float(kv.x << 16), __uint_as_float(kv.x & 0xFFFF0000u),
                         __uint_as_float(kv.y << 16), __uint_as_float(kv.y & 0xFFFF0000u)};
    float m = fmaxf(fmaxf(fabsf(kk[0]), fabsf(kk[1])), fmaxf(fabsf(kk[2]), fabsf(kk[3])));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));   // over the block's 8 lanes
    const int e = m > 0.f ? min(max(ilogbf(m) - 2 + 127, 0), 254) : 0;
    const float mul = __uint_as_float(static_cast<uint32_t>(254 - e) << 23);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = __nv_cvt_float_to_fp4(kk[i] * mul, __NV_E2M1, cudaRoundNearest) & 0xFu;
    int64_t row = 0;
    int slot = 0;
    if (new_token_slot(p.b, p.pool, t, p.status, row, slot)) {
      uint8_t* page = p.pool_w + row * p.pool.row_stride + p.pool.idx_off;
      *reinterpret_cast<uint16_t*>(page + slot * (kIdxDim / 2) + 2 * lane) =
          static_cast<uint16_t>(c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12));
      if ((lane & 7) == 0) page[static_cast<int64_t>(p.pool.bs) * (kIdxDim / 2) + slot * 4 + (lane >> 3)] = static_cast<uint8_t>(e);
    }
  } else if (p.k_new && blockIdx.x == 1 && warp < nt) {
    const int t = t0 + warp;
    const uint2 kv = __ldg(reinterpret_cast<const uint2*>(p.k_new + static_cast<int64_t>(t) * kIdxDim) + lane);
    const float k0 = __uint_as_float(kv.x << 16), k1 = __uint_as_float(kv.x & 0xFFFF0000u);
    const float k2 = __uint_as_float(kv.y << 16), k3 = __uint_as_float(kv.y & 0xFFFF0000u);
    float m = fmaxf(fmaxf(fabsf(k0), fabsf(k1)), fmaxf(fabsf(k2), fabsf(k3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = m > 0.f ? m / 448.0f : 1.0f;
    int64_t row = 0;
    int slot = 0;
    if (new_token_slot(p.b, p.pool, t, p.status, row, slot)) {
      uint8_t* page = p.pool_w + row * p.pool.row_stride + p.pool.idx_off;
      *reinterpret_cast<uint32_t*>(page + slot * kIdxDim + 4 * lane) = f4_to_e4m3x4(k0 / s, k1 / s, k2 / s, k3 / s);
      if (lane == 0) *reinterpret_cast<float*>(page + static_cast<int64_t>(p.pool.bs) * kIdxDim + slot * 4) = s;
    }
  }
  if (quarter == 0) cluster_arrive_relaxed();
  cluster_wait();   // no CTA leaves while the first may still read its sums
  // no copy or MMA outlives the CTA (after a timeout some may still run)
  if (warp == PROD_WARP && lane == 0)
    for (int c = max(0, issued - RING); c < issued; ++c) drain_wait(&full[c % RING], (c / RING) & 1);
  if (warp == MMA_WARP && lane == 0) drain_wait(done, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) tmem_dealloc(tmem, 32);
}

// The new tokens' latents into their cache slots: one CTA of 64 threads per
// token, thread i < 36 takes values 16 i .. 16 i + 15.
__global__ void __launch_bounds__(64) write_latent_kernel(LatentWriteParams p) {
  const int t = blockIdx.x, i = threadIdx.x;
  grid_dep_wait();
  __shared__ int64_t row_sh;
  __shared__ int slot_sh, ok_sh;
  if (i == 0) {
    int64_t row = 0;
    int slot = 0;
    ok_sh = new_token_slot(p.b, p.pool, t, p.status, row, slot) ? 1 : 0;
    row_sh = row;
    slot_sh = slot;
  }
  __syncthreads();
  if (!ok_sh || i >= 36) return;
  const uint4* src = reinterpret_cast<const uint4*>(p.latent + static_cast<int64_t>(t) * kLatDim + 16 * i);
  const uint4 a = __ldg(src), b = __ldg(src + 1);
  const uint32_t w8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float v[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[2 * j] = __uint_as_float(w8[j] << 16);
    v[2 * j + 1] = __uint_as_float(w8[j] & 0xFFFF0000u);
  }
  uint8_t* page = p.pool_w + row_sh * p.pool.row_stride + p.pool.lat_off;
  if (p.pool.lat_fmt == DSA_LAT_FP8) {
    uint4 o;
    o.x = f4_to_e4m3x4(v[0], v[1], v[2], v[3]);
    o.y = f4_to_e4m3x4(v[4], v[5], v[6], v[7]);
    o.z = f4_to_e4m3x4(v[8], v[9], v[10], v[11]);
    o.w = f4_to_e4m3x4(v[12], v[13], v[14], v[15]);
    *reinterpret_cast<uint4*>(page + static_cast<int64_t>(slot_sh) * kLatDim + 16 * i) = o;
    return;
  }
  // NVFP4: scale e4m3(max|x| / 6), values e2m1(x / scale) (zeros for a zero scale)
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
  const __nv_fp8_storage_t scode = __nv_cvt_float_to_fp8(m / 6.0f, __NV_SATFINITE, __NV_E4M3);
  const __half_raw shr = __nv_cvt_fp8_to_halfraw(scode, __NV_E4M3);
  const float sv = __half2float(*reinterpret_cast<const __half*>(&shr));
  uint32_t packed[2] = {0u, 0u};
  if (sv > 0.f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = static_cast<uint32_t>(
          __nv_cvt_float2_to_fp4x2(make_float2(v[2 * j] / sv, v[2 * j + 1] / sv), __NV_E2M1, cudaRoundNearest));
      packed[j >> 2] |= (byte & 0xFFu) << (8 * (j & 3));
    }
  }
  uint8_t* rec = page + static_cast<int64_t>(slot_sh) * 352;
  *reinterpret_cast<uint2*>(rec + 8 * i) = make_uint2(packed[0], packed[1]);
  rec[288 + i] = static_cast<uint8_t>(scode);
  if (i < 7) *reinterpret_cast<uint32_t*>(rec + 324 + 4 * i) = 0u;
}

cudaError_t launch_indexer_front(const CUtensorMap& wmap, const FrontParams& p, cudaStream_t st) {
  cudaError_t e = set_func_attr_once(reinterpret_cast<const void*>(indexer_front_kernel),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, front::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const dim3 grid(kIdxHeads * 4, static_cast<unsigned>(cdiv(p.b.T, front::CHUNK)));
  return launch_ex(indexer_front_kernel, grid, dim3(front::THREADS), front::SMEM_BYTES, st, false, 4u, wmap, p);
}

cudaError_t launch_write_latent(const LatentWriteParams& p, cudaStream_t st) {
  return launch_ex(write_latent_kernel, dim3(p.b.T), dim3(64), 0, st, false, 0u, p);
}

}  // namespace dsa

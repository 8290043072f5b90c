// front.cu — the fused indexer front and the new tokens' cache writes.
//
// vLLM K3.1 Pro day-0 post, "Low-latency decode: a fused DSA decode path": "a
// fused indexer front: the query norm, the indexer's query projection, its FP8
// or MXFP4 quantization with the head weights folded in, and the new token's
// index key, in one kernel"; the MLA query kernel "writing the new token's
// latent into the KV cache".  Readings (the post prints no shapes): RMSNorm over
// the compressed query of width d_q, q = W . norm(c_q) with W [32 * 128, d_q],
// FP8 per (token, head) with s = max|q_h| / 448 folded into the head weight,
// the new key FP8 with s_k = max|k| / 448, latents FP8 (plain e4m3) or NVFP4
// (e4m3 scale max|x| / 6 per 16 values, e2m1 values).
//
// Indexer front.  At decode the projection is a weight stream (4096 x d_q bf16,
// 12.6 MB at d_q = 1536) against a few queries, so it runs on the CUDA cores as a
// blocked GEMV, not on the tensor cores (a tile of 8 tokens would leave them
// idle and the fp32 query would need two bf16 terms).  Grid (4 quarters x 32
// heads, token chunks of 8) in clusters of the 4 quarters of a head.  Each CTA
// brings its 32 rows of W into a 4-slot ring by TMA, 256 dims a copy, while 8
// warps normalise the chunk's queries into shared memory (fp32).  Thread (row
// group g, lane kl of 128) accumulates 8 rows x 8 tokens over dims 2kl, 2kl + 1
// of every 256-dim chunk with packed fp32 FMAs; the 128 partial sums of each
// output are reduced by a butterfly inside the warps (each lane ends with 2 of
// its warp's 64 outputs) and across the 4 warps of the group in shared memory.
// The head's maximum comes from the four CTAs through distributed shared memory,
// then each CTA quantizes its rows.  The first CTA of the first head also writes
// the chunk's new index keys into their cache slots.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "../../include/dsa.h"
#include "params.cuh"

namespace dsa {

namespace front {
constexpr int THREADS = 512;
constexpr int CHUNK = 8;                 // query tokens per CTA
constexpr int ROWS = 32;                 // output rows (dims of one head) per CTA
constexpr int MAX_DQ = 4096;
constexpr int KBOX = 256;                // dims of W per copy
constexpr int RING = 4;                  // copies in flight
constexpr int SLOT_BYTES = ROWS * KBOX * 2;
// dynamic shared memory: ring | y [CHUNK][y_pitch] fp32 | red [16 warps][64] | qv [ROWS][CHUNK] |
// amax [CHUNK] x 2 | bars [RING] | abort flag
__host__ __device__ constexpr int y_pitch(int dq) { return (dq + KBOX - 1) / KBOX * KBOX; }
__host__ __device__ constexpr int smem_bytes(int dq) {
  return RING * SLOT_BYTES + CHUNK * y_pitch(dq) * 4 + 16 * 64 * 4 + ROWS * CHUNK * 4 + 2 * CHUNK * 4 + RING * 8 + 16 +
         128;
}
static_assert(smem_bytes(MAX_DQ) <= 232448, "front shared memory");
}  // namespace front

// d = a * b + c on two fp32 lanes at once (one packed FMA, round to nearest)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&d);
}

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
  uint8_t* fsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fsm_raw) + 127) & ~uintptr_t(127));
  const int dq = p.d_q;
  const int ypitch = y_pitch(dq);
  const int nk = ypitch / KBOX;                                       // 256-dim chunks of W
  const int kbox = dq < KBOX ? dq : KBOX;                             // dims per copy
  uint8_t* ring = fsm;                                                // [RING][ROWS][kbox] bf16
  float* y = reinterpret_cast<float*>(fsm + RING * SLOT_BYTES);       // [CHUNK][ypitch] normalised queries
  float* red = y + CHUNK * ypitch;                                    // [16 warps][64] partial sums
  float* qv = red + 16 * 64;                                          // [ROWS][CHUNK] projections of this CTA
  float* amax_sh = qv + ROWS * CHUNK;                                 // [CHUNK] this CTA's per-token max |q|
  float* amax_all = amax_sh + CHUNK;                                  // [CHUNK] the head's
  uint64_t* bars = reinterpret_cast<uint64_t*>(amax_all + CHUNK);     // [RING]
  int* abortf = reinterpret_cast<int*>(bars + RING);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = blockIdx.x & 3, h = blockIdx.x >> 2;
  const int row0 = h * 128 + quarter * ROWS;
  const int t0 = blockIdx.y * CHUNK;
  const int nt = min(CHUNK, p.b.T - t0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < RING; ++i) mbar_init(&bars[i], 1);
    *abortf = 0;
    fence_mbar_init();
    prefetch_tensormap(&wmap);
  }
  __syncthreads();
  grid_dep_wait();
  // 1. the first W copies, then RMSNorm of each token of the chunk (one warp per
  // token; y past d_q and the rows of absent tokens are zero)
  if (threadIdx.x == 0)
    for (int c = 0; c < RING && c < nk; ++c) {
      mbar_arrive_expect_tx(&bars[c], ROWS * kbox * 2);
      tma_load_2d(ring + c * SLOT_BYTES, &wmap, &bars[c], c * KBOX, row0);
    }
  if (warp < CHUNK) {
    float* yt = y + warp * ypitch;
    if (warp < nt) {
      const __nv_bfloat16* x = p.c_q + static_cast<int64_t>(t0 + warp) * dq;
      float ss = 0.f;
      for (int i = lane * 8; i < dq; i += 256) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + i));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float o8[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          o8[2 * j] = __uint_as_float(w4[j] << 16);
          o8[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
          ss = fmaf(o8[2 * j], o8[2 * j], fmaf(o8[2 * j + 1], o8[2 * j + 1], ss));
        }
        reinterpret_cast<float4*>(yt + i)[0] = make_float4(o8[0], o8[1], o8[2], o8[3]);
        reinterpret_cast<float4*>(yt + i)[1] = make_float4(o8[4], o8[5], o8[6], o8[7]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float r = 1.0f / sqrtf(ss / static_cast<float>(dq) + p.eps);
      __syncwarp();
      for (int i = lane * 8; i < dq; i += 256) {
        const uint4 gm = __ldg(reinterpret_cast<const uint4*>(p.gamma + i));
        const uint32_t g4[4] = {gm.x, gm.y, gm.z, gm.w};
        float4* dst = reinterpret_cast<float4*>(yt + i);
        float4 a = dst[0], c = dst[1];
        a.x = a.x * r * __uint_as_float(g4[0] << 16);
        a.y = a.y * r * __uint_as_float(g4[0] & 0xFFFF0000u);
        a.z = a.z * r * __uint_as_float(g4[1] << 16);
        a.w = a.w * r * __uint_as_float(g4[1] & 0xFFFF0000u);
        c.x = c.x * r * __uint_as_float(g4[2] << 16);
        c.y = c.y * r * __uint_as_float(g4[2] & 0xFFFF0000u);
        c.z = c.z * r * __uint_as_float(g4[3] << 16);
        c.w = c.w * r * __uint_as_float(g4[3] & 0xFFFF0000u);
        dst[0] = a;
        dst[1] = c;
      }
      for (int i = dq + lane; i < ypitch; i += 32) yt[i] = 0.f;
    } else {
      for (int i = lane; i < ypitch; i += 32) yt[i] = 0.f;
    }
  }
  __syncthreads();
  // 2. thread (group g of 8 rows, kl of 128) over dims 2 kl, 2 kl + 1 of each chunk
  const int g = warp >> 2, kl = ((warp & 3) << 5) | lane;
  float2 acc[8][CHUNK / 2];   // [row][token pair]
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int t = 0; t < CHUNK / 2; ++t) acc[i][t] = make_float2(0.f, 0.f);
  const Abort ab{abortf, p.status};
  bool ok = true;
#pragma unroll 1
  for (int c = 0; c < nk; ++c) {
    const int slot = c % RING;
    if (ok) ok = mbar_wait(&bars[slot], (c / RING) & 1, ab);
    if (ok && 2 * kl < kbox) {
      const uint8_t* wsl = ring + slot * SLOT_BYTES + (8 * g) * (kbox * 2) + 4 * kl;
      float2 w2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(wsl + i * (kbox * 2));
        w2[i] = make_float2(__uint_as_float(wb << 16), __uint_as_float(wb & 0xFFFF0000u));
      }
      const float* yc = y + c * KBOX + 2 * kl;
#pragma unroll
      for (int tp = 0; tp < CHUNK / 2; ++tp) {
        const float2 ya = *reinterpret_cast<const float2*>(yc + (2 * tp) * ypitch);       // token 2tp, dims d, d+1
        const float2 yb = *reinterpret_cast<const float2*>(yc + (2 * tp + 1) * ypitch);   // token 2tp+1
        const float2 y0 = make_float2(ya.x, yb.x), y1 = make_float2(ya.y, yb.y);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[i][tp] = ffma2(make_float2(w2[i].x, w2[i].x), y0, acc[i][tp]);
          acc[i][tp] = ffma2(make_float2(w2[i].y, w2[i].y), y1, acc[i][tp]);
        }
      }
    }
    __syncthreads();   // every warp is done with this slot
    if (threadIdx.x == 0 && c + RING < nk && !*reinterpret_cast<volatile int*>(abortf)) {
      mbar_arrive_expect_tx(&bars[slot], ROWS * kbox * 2);
      tma_load_2d(ring + slot * SLOT_BYTES, &wmap, &bars[slot], (c + RING) * KBOX, row0);
    }
  }
  // 3. reduce each output's 128 partial sums: a butterfly over the lanes leaves lane l
  // with outputs 2l, 2l + 1 (output v = row * 8 + token) of the warp, then the 4 warps
  // of the group add in shared memory
  float v[64];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int tp = 0; tp < CHUNK / 2; ++tp) {
      v[i * 8 + 2 * tp] = acc[i][tp].x;
      v[i * 8 + 2 * tp + 1] = acc[i][tp].y;
    }
#pragma unroll
  for (int o = 16, n = 64; o > 0; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = upper ? v[j] : v[j + n / 2];
      const float keep = upper ? v[j + n / 2] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  red[warp * 64 + 2 * lane] = v[0];
  red[warp * 64 + 2 * lane + 1] = v[1];
  __syncthreads();
  if (threadIdx.x < ROWS * CHUNK) {
    const int r = threadIdx.x >> 3, t = threadIdx.x & 7;   // row of the CTA, token
    const int gg = r >> 3, vi = (r & 7) * 8 + t;
    float sum = 0.f;
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) sum += red[(gg * 4 + w4) * 64 + vi];
    qv[r * CHUNK + t] = sum;
  }
  __syncthreads();
  // 4. the head's max |q| per token: this CTA's 32 rows, then the cluster's four quarters
  if (threadIdx.x < CHUNK) {
    float m = 0.f;
    for (int rr = 0; rr < ROWS; ++rr) m = fmaxf(m, fabsf(qv[rr * CHUNK + threadIdx.x]));
    amax_sh[threadIdx.x] = m;
  }
  cluster_arrive();
  cluster_wait();
  if (threadIdx.x < CHUNK) {
    float m = 0.f;
    for (uint32_t r = 0; r < 4; ++r)
      m = fmaxf(m, __uint_as_float(ld_cluster_u32(cluster_map(smem_u32(&amax_sh[threadIdx.x]), r))));
    amax_all[threadIdx.x] = m;
  }
  cluster_arrive_relaxed();   // done reading the other quarters
  __syncthreads();
  // 5. codes e4m3(q / s), s = max / 448 (1 for an all-zero head); folded weights by quarter 0
  if (threadIdx.x < CHUNK * ROWS / 4) {
    const int t = threadIdx.x / (ROWS / 4), r4 = (threadIdx.x % (ROWS / 4)) * 4;   // 4 rows per thread
    if (t < nt) {
      const float m = amax_all[t];
      const float s = m > 0.f ? m / 448.0f : 1.0f;
      const uint32_t code = f4_to_e4m3x4(qv[(r4 + 0) * CHUNK + t] / s, qv[(r4 + 1) * CHUNK + t] / s,
                                         qv[(r4 + 2) * CHUNK + t] / s, qv[(r4 + 3) * CHUNK + t] / s);
      *reinterpret_cast<uint32_t*>(p.q_idx + (static_cast<int64_t>(t0 + t) * kIdxHeads + h) * kIdxDim + quarter * ROWS +
                                   r4) = code;
      if (quarter == 0 && r4 == 0) p.w_out[static_cast<int64_t>(t0 + t) * kIdxHeads + h] = p.head_w[(t0 + t) * kIdxHeads + h] * s;
    }
  }
  // 6. the chunk's new index keys (first quarter of head 0): one warp per token,
  // four values per lane, s_k = max |k| / 448 in fp32
  if (p.k_new && blockIdx.x == 0 && warp < nt) {
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
  cluster_wait();   // no CTA leaves while another may still read its maxima
  // no copy into shared memory outlives the CTA (the last copy of each slot)
  if (threadIdx.x < RING && static_cast<int>(threadIdx.x) < nk)
    drain_wait(&bars[threadIdx.x], ((nk - 1 - static_cast<int>(threadIdx.x)) / RING) & 1);
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
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, front::smem_bytes(front::MAX_DQ));
  if (e != cudaSuccess) return e;
  const dim3 grid(kIdxHeads * 4, static_cast<unsigned>(cdiv(p.b.T, front::CHUNK)));
  return launch_ex(indexer_front_kernel, grid, dim3(front::THREADS), front::smem_bytes(p.d_q), st, false, 4u, wmap,
                   p);
}

cudaError_t launch_write_latent(const LatentWriteParams& p, cudaStream_t st) {
  return launch_ex(write_latent_kernel, dim3(p.b.T), dim3(64), 0, st, false, 0u, p);
}

}  // namespace dsa

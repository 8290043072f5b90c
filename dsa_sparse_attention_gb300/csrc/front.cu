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
// GEMV, not on the tensor cores.  Grid (4 quarters x 32 heads, token chunks of 8)
// in clusters of the 4 quarters of a head: each CTA normalises its chunk's
// queries into shared memory (fp32), streams its 32 rows of W once (16-byte
// loads, all of a row's loads in flight) and keeps the 32 x T dot products; the
// head's maximum comes from the four CTAs through distributed shared memory,
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

__global__ void __launch_bounds__(front::THREADS) indexer_front_kernel(FrontParams p) {
  using namespace front;
  extern __shared__ __align__(16) float fsm[];
  float* y = fsm;                                     // [CHUNK][d_q] normalised queries
  float* qv = fsm + CHUNK * p.d_q;                    // [ROWS][CHUNK] projections of this CTA
  float* amax_sh = qv + ROWS * CHUNK;                 // [CHUNK] this CTA's per-token max |q|
  float* amax_all = amax_sh + CHUNK;                  // [CHUNK] the head's
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = blockIdx.x & 3, h = blockIdx.x >> 2;
  const int t0 = blockIdx.y * CHUNK;
  const int nt = min(CHUNK, p.b.T - t0);
  const int dq = p.d_q;
  grid_dep_wait();
  // 1. RMSNorm of each token of the chunk (one warp per token)
  if (warp < nt) {
    const __nv_bfloat16* x = p.c_q + static_cast<int64_t>(t0 + warp) * dq;
    float ss = 0.f;
    for (int i = lane * 8; i < dq; i += 256) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + i));
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = __uint_as_float(w4[j] << 16), c = __uint_as_float(w4[j] & 0xFFFF0000u);
        ss = fmaf(a, a, fmaf(c, c, ss));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(dq) + p.eps);
    for (int i = lane * 8; i < dq; i += 256) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + i));
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(p.gamma + i));
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w}, g4[4] = {g.x, g.y, g.z, g.w};
      float o8[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o8[2 * j] = __uint_as_float(w4[j] << 16) * r * __uint_as_float(g4[j] << 16);
        o8[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u) * r * __uint_as_float(g4[j] & 0xFFFF0000u);
      }
      float4* dst = reinterpret_cast<float4*>(y + warp * dq + i);
      dst[0] = make_float4(o8[0], o8[1], o8[2], o8[3]);
      dst[1] = make_float4(o8[4], o8[5], o8[6], o8[7]);
    }
  }
  __syncthreads();
  // 2. this CTA's 32 rows (dims 32 quarter .. of head h), two per warp; lane l takes
  // the 16-byte pieces l, l + 32, ... of a row (d_q / 8 pieces)
  for (int rr = warp; rr < ROWS; rr += THREADS / 32) {
    const int row = h * 128 + quarter * ROWS + rr;
    const uint4* wrow = reinterpret_cast<const uint4*>(p.w_qi + static_cast<int64_t>(row) * dq);
    const int npc = dq / 8;
    float acc[CHUNK];
#pragma unroll
    for (int t = 0; t < CHUNK; ++t) acc[t] = 0.f;
    for (int base = 0; base < npc; base += 32 * 8) {
      uint4 wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {   // up to eight pieces of the row in flight per lane
        const int pc = base + lane + 32 * u;
        wv[u] = pc < npc ? __ldg(wrow + pc) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int pc = base + lane + 32 * u;
        if (pc >= npc) break;
        const uint32_t w4[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
        float wf[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          wf[2 * j] = __uint_as_float(w4[j] << 16);
          wf[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
        }
#pragma unroll
        for (int t = 0; t < CHUNK; ++t) {
          if (t >= nt) break;
          const float4 a = *reinterpret_cast<const float4*>(y + t * dq + pc * 8);
          const float4 c = *reinterpret_cast<const float4*>(y + t * dq + pc * 8 + 4);
          float s = acc[t];
          s = fmaf(wf[0], a.x, s);
          s = fmaf(wf[1], a.y, s);
          s = fmaf(wf[2], a.z, s);
          s = fmaf(wf[3], a.w, s);
          s = fmaf(wf[4], c.x, s);
          s = fmaf(wf[5], c.y, s);
          s = fmaf(wf[6], c.z, s);
          s = fmaf(wf[7], c.w, s);
          acc[t] = s;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < CHUNK; ++t) {
      float s = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) qv[rr * CHUNK + t] = s;
    }
  }
  __syncthreads();
  // 3. the head's max |q| per token: this CTA's 32 rows, then the cluster's four quarters
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
  // 4. codes e4m3(q / s), s = max / 448 (1 for an all-zero head); folded weights by quarter 0
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
  // 5. the chunk's new index keys (first quarter of head 0): one warp per token,
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

cudaError_t launch_indexer_front(const FrontParams& p, cudaStream_t st) {
  const size_t smem = (static_cast<size_t>(front::CHUNK) * p.d_q + front::ROWS * front::CHUNK + 2 * front::CHUNK) * 4;
  cudaError_t e = set_func_attr_once(reinterpret_cast<const void*>(indexer_front_kernel),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(kIdxHeads * 4, static_cast<unsigned>(cdiv(p.b.T, front::CHUNK)));
  return launch_ex(indexer_front_kernel, grid, dim3(front::THREADS), smem, st, false, 4u, p);
}

cudaError_t launch_write_latent(const LatentWriteParams& p, cudaStream_t st) {
  return launch_ex(write_latent_kernel, dim3(p.b.T), dim3(64), 0, st, false, 0u, p);
}

}  // namespace dsa

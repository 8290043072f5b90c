// mla_q.cuh — the absorbed query of one MLA head as two e4m3 terms, laid out as
// the FP8 attention kernel's tensor-core operand.
//
// vLLM K3.1 Pro day-0 post, "Sparse Attention in K3.1 Pro": MLA attends with 96
// absorbed query heads over 576-dim latents; the latents are FP8 ("KV cache
// footprint").  To multiply the bf16 query with e4m3 latents on the FP8 tensor
// cores without rounding it, each head's 576 values are scaled by a power of two
// 2^k (chosen so the largest |q| lands in [224, 448]) and split into
// hi = e4m3(2^k q) and lo = e4m3(2^k q - hi).  A bf16 value has 8 significant
// bits and an e4m3 value 4, so hi + lo = 2^k q exactly whenever |2^k q| >= 1/4
// (smaller values keep an absolute error of at most 2^-10 / 2^k).
//
// Layout of one token's terms (110,592 bytes, then 96 int32 exponents k):
// nine K-chunks of [96 heads x 128 bytes], each already in the tensor core's
// 128-byte-swizzled K-major order (the 16-byte piece j of head row h sits at
// piece j ^ (h % 8)), so a plain bulk copy into 1024-byte-aligned shared memory
// yields the MMA operand.  Chunks: hi dims 0..511 (chunks 0..3, 128 dims each),
// [hi dims 512..575 | lo dims 512..575] (chunk 4), lo dims 0..511 (chunks 5..8).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace dsa {

constexpr int kQChunkBytes = kMlaHeads * 128;               // one K-chunk: 12,288 B
constexpr int kQChunks = 9;
constexpr int kQTermBytes = kQChunks * kQChunkBytes;        // 110,592 B
constexpr int kQTokenBytes = kQTermBytes + kMlaHeads * 4;   // + exponents: 110,976 B (a multiple of 16)

// Two floats -> two e4m3 codes (round to nearest even, saturating), element 0 in the low byte.
__device__ __forceinline__ uint32_t f2_to_e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xFFFFu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// log2 of the power-of-two scale that puts amax in [224, 448] (0 for a zero or
// subnormal amax).
__device__ __forceinline__ int q_scale_log2(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int e = static_cast<int>((b >> 23) & 0xFF) - 127;
  if ((b & 0x7FFFFFFFu) == 0 || e < -126) return 0;
  const bool above = (b & 0x7FFFFFu) > 0x600000u;   // mantissa above 1.75
  const int k = (above ? 7 : 8) - e;
  return k < -126 ? -126 : (k > 126 ? 126 : k);
}

// One warp: head h of query q_tok (bf16 [96][576]) -> its rows of the nine
// chunks at `terms` (a token's 110,592 bytes, global or shared) and its exponent.
// Lane l takes the 16-byte pieces l, l + 32 and l + 64 (dims 8 piece .. + 7).
__device__ __forceinline__ void q_head_to_terms(const __nv_bfloat16* q_tok, int h, uint8_t* terms, int32_t* exps) {
  const int lane = threadIdx.x & 31;
  const uint4* src = reinterpret_cast<const uint4*>(q_tok + static_cast<int64_t>(h) * kLatDim);
  uint4 v[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int pc = lane + 32 * r;
    v[r] = pc < 72 ? __ldg(src + pc) : make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t am = 0;   // |q| bits: non-negative floats order as unsigned integers
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const uint32_t w4[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) am = max(am, max((w4[j] << 16) & 0x7FFFFFFFu, w4[j] & 0x7FFF0000u));
  }
  const int k2 = q_scale_log2(__uint_as_float(__reduce_max_sync(0xffffffffu, am)));
  const float sc = __uint_as_float(static_cast<uint32_t>(k2 + 127) << 23);
  if (lane == 0) exps[h] = k2;
  uint8_t* row = terms + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int pc = lane + 32 * r;
    if (pc >= 72) break;
    const uint32_t w4[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
    uint32_t hi[2], lo[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {   // 4 values -> 4 bytes of each term
      const float a0 = __uint_as_float(w4[2 * j] << 16) * sc;
      const float a1 = __uint_as_float(w4[2 * j] & 0xFFFF0000u) * sc;
      const float a2 = __uint_as_float(w4[2 * j + 1] << 16) * sc;
      const float a3 = __uint_as_float(w4[2 * j + 1] & 0xFFFF0000u) * sc;
      const uint32_t h01 = f2_to_e4m3x2(a0, a1), h23 = f2_to_e4m3x2(a2, a3);
      const float2 b01 = e4m3x2_to_f2(h01), b23 = e4m3x2_to_f2(h23);
      hi[j] = h01 | (h23 << 16);
      lo[j] = f2_to_e4m3x2(a0 - b01.x, a1 - b01.y) | (f2_to_e4m3x2(a2 - b23.x, a3 - b23.y) << 16);
    }
    const int G = pc >> 1, half8 = (pc & 1) * 8;   // 16-dim group, byte offset inside its 16-byte piece
    const int hc = G < 32 ? (G >> 3) : 4, hi_i = G < 32 ? (G & 7) : (G - 32);
    const int lc = G < 32 ? 5 + (G >> 3) : 4, lo_i = G < 32 ? (G & 7) : (G - 28);
    *reinterpret_cast<uint2*>(row + hc * kQChunkBytes + ((hi_i ^ (h & 7)) << 4) + half8) = make_uint2(hi[0], hi[1]);
    *reinterpret_cast<uint2*>(row + lc * kQChunkBytes + ((lo_i ^ (h & 7)) << 4) + half8) = make_uint2(lo[0], lo[1]);
  }
}

}  // namespace dsa

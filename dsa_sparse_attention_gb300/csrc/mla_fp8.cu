// mla_fp8.cu — sparse MLA over FP8 latents with the latents read once, straight
// into the tensor cores' operand tiles, and the splits of a token reduced inside
// a thread-block cluster.
//
// vLLM K3.1 Pro day-0 post, "Sparse Attention in K3.1 Pro" (+ Figure 1): every
// query head attends exactly over only the selected tokens' 576-byte FP8
// latents ("KV cache footprint"); 96 absorbed query heads, value = first 512
// latent dims, NoPE ("What's new in Kimi K3.1 Pro").  Partial results of the
// splits of the selection are merged by log-sum-exp, as the post's DCP section
// merges partial outputs across GPUs ("Long context: decode context
// parallelism with a sparse indexer"); here the splits are the CTAs of a
// cluster and the merge runs through distributed shared memory.
//
// One CTA per (query token, 128 selected tokens); the nsplit CTAs of a token
// form one cluster.  Per CTA:
//  1. The 128 selected latent records (576 B each) are gathered with 16-byte
//     cp.async copies directly into five 128-byte-swizzled K-chunks of
//     [128 tokens x 128 B] (dims 0..511 in chunks 0..3; chunk 4 holds dims
//     512..575 twice, see 2).  No conversion: e4m3 is the MMA's operand type.
//  2. While those copies fly, the query [96 heads x 576] bf16 is split per head
//     into two e4m3 terms: with a power-of-two scale s_h putting the head's
//     largest |q| in [224, 448], hi = e4m3(s_h q) and lo = e4m3(s_h q - hi).  A
//     bf16 value has 8 significant bits and each e4m3 term holds 4, so hi + lo
//     equals s_h q exactly for every |s_h q| >= 1/4 (below that the error is at
//     most 2^-10 / s_h).  K-chunks of the query operand: hi dims 0..511 (four
//     chunks), [hi 512..575 | lo 512..575] (chunk 4), lo dims 0..511.
//  3. S[head, token] = sum_k q_term[head, k] . latent[token, k] over the nine
//     chunks: tcgen05.mma kind::f8f6f4, M = 128 (heads 0..95; lanes 96..127 are
//     padding nobody reads), N = 128 tokens, K = 1152, fp32 in TMEM.  Heads on
//     TMEM lanes make the softmax thread-local: four threads per head, 32
//     tokens each.
//  4. p = 2^(logit2 - max + 8) is rounded once to fp16 (11 significant bits),
//     then split exactly into three e4m3 terms (4 + 4 + 3 bits), written as
//     three K-major [96 heads x 128 tokens] operand tiles; the row sum is the
//     sum of the same fp16 values, so the normalisation matches the weights.
//  5. O^T[dim, head] += V^T[dim, token] . P^T[token, head] for the four 128-dim
//     blocks of the value, three terms each: M = 128 dims, N = 96 heads, K =
//     3 x 128; A is the gathered latent tile itself read MN-major (the same
//     bytes as step 3's B operand), B the P tiles.  TMEM: S in columns
//     [0, 128), O^T blocks at 128 + 96 v: 512 columns.
//  6. One split: O / l in bf16.  Several: each CTA stores its normalised fp16
//     partial and its per-head (max, sum) in its own shared memory; after one
//     cluster barrier, CTA r sums the 32-dim blocks b with b % nsplit == r over
//     all CTAs of the cluster (weights 2^(m_j - M) l_j / L) and writes them;
//     rank 0 writes lse.  A second barrier keeps every CTA alive until the
//     others have read it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>
#include <vector>

#include "params.cuh"

namespace dsa {

namespace mla8 {
constexpr int THREADS = 512;                      // 16 warps
constexpr int QCHUNK = 96 * 128;                  // one K-chunk of the query operand (12 KB)
constexpr int NQCHUNK = 9;
constexpr int LCHUNK = 128 * 128;                 // one K-chunk of the latent tile (16 KB)
constexpr int NLCHUNK = 5;
constexpr int OFF_Q = 0;                          // query terms; later P, then the fp16 partial
constexpr int OFF_LAT = NQCHUNK * QCHUNK;         // 110,592: latent tile; after PV the merge scratch
constexpr int OFF_SMALL = OFF_LAT + NLCHUNK * LCHUNK;   // 192,512
constexpr int OFF_SRC = OFF_SMALL;                // [128] int64 byte offset of each selected record (-1: absent)
constexpr int OFF_QEXP = OFF_SRC + 128 * 8;       // [96] int: log2 of the query scale of each head
constexpr int OFF_REDM = OFF_QEXP + 96 * 4;       // [4][96] float: tile max per token quarter
constexpr int OFF_REDL = OFF_REDM + 4 * 96 * 4;   // [4][96] float: sum per token quarter
constexpr int OFF_ML = OFF_REDL + 4 * 96 * 4;     // [96] float2: this CTA's (max, sum), read by the cluster
constexpr int OFF_INV = OFF_ML + 96 * 8;          // [96] float: 1 / sum
constexpr int OFF_BARS = OFF_INV + 96 * 4;
constexpr int OFF_MISC = OFF_BARS + 8 * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
constexpr int P_TERM = 96 * 128;                  // one e4m3 term of P^T (12 KB), at OFF_Q
constexpr int STG_PITCH = 208;                    // fp16 partial row: 96 heads (192 B) + padding
constexpr int OFF_WGT = OFF_LAT;                  // merge: [16][96] float weights
constexpr int OFF_TILE = OFF_LAT + 16 * 96 * 4;   // merge: [96 heads][32 dims] bf16
constexpr int MAX_SPLITS = 16;
constexpr int S_COL = 0;
constexpr int O_COL = 128;
constexpr int MMA_WARP = 3;                       // a warp of lane quarter 3, which has no softmax role
static_assert(OFF_LAT % 1024 == 0 && OFF_SMALL % 1024 == 0, "operand tiles are 1024-byte aligned");
static_assert(3 * P_TERM <= OFF_LAT, "P fits the query region");
static_assert(kVDim * STG_PITCH <= OFF_LAT, "the fp16 partial fits the query region");
static_assert(OFF_TILE + 96 * 32 * 2 <= OFF_SMALL, "merge scratch fits the latent region");
static_assert(SMEM_BYTES <= 232448, "shared memory");
}  // namespace mla8

__device__ __forceinline__ uint8_t* align1024_m8(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// 16-byte global -> shared copy (cp.async, L2 only); src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Two floats -> two e4m3 codes (round to nearest even, saturating), element 0 in the low byte.
__device__ __forceinline__ uint32_t f2_to_e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xFFFFu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
__device__ __forceinline__ uint32_t h2_to_e4m3x2(__half2 v) {
  return static_cast<uint32_t>(
      __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&v), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ __half2 e4m3x2_to_h2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xFFFFu), __NV_E4M3);
  return *reinterpret_cast<const __half2*>(&h);
}

// 2^x on the multi-function unit (relative error about 2^-22; subnormal results flush to 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2 of the power-of-two scale that puts amax in [224, 448] (0 for amax = 0).
__device__ __forceinline__ int q_scale_log2(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int e = static_cast<int>((b >> 23) & 0xFF) - 127;
  if ((b & 0x7FFFFFFFu) == 0 || e < -126) return 0;          // zero or subnormal maximum: leave unscaled
  const bool above = (b & 0x7FFFFFu) > 0x600000u;            // mantissa above 1.75
  int k = (above ? 7 : 8) - e;
  return k < -126 ? -126 : (k > 126 ? 126 : k);
}

template <int DUMMY>
__global__ void __launch_bounds__(mla8::THREADS, 1) sparse_mla_fp8_kernel(MlaParams p) {
  using namespace mla8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024_m8(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* ready = bars + 0;    // the latent tile and the query terms are in shared memory (512 arrivals)
  uint64_t* s_full = bars + 1;   // QK done
  uint64_t* p_full = bars + 2;   // P written (12 softmax warps)
  uint64_t* o_done = bars + 3;   // PV done
  uint64_t* drain = bars + 4;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* abortf = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  int* has_work = reinterpret_cast<int*>(smem + OFF_MISC + 16);
  int64_t* src_off = reinterpret_cast<int64_t*>(smem + OFF_SRC);
  int* qexp = reinterpret_cast<int*>(smem + OFF_QEXP);
  float* red_m = reinterpret_cast<float*>(smem + OFF_REDM);
  float* red_l = reinterpret_cast<float*>(smem + OFF_REDL);
  float2* ml = reinterpret_cast<float2*>(smem + OFF_ML);
  float* inv_l = reinterpret_cast<float*>(smem + OFF_INV);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int t = blockIdx.y;
  const int split = blockIdx.x;   // = rank in the cluster (cluster dims = (nsplit, 1, 1))
  const int nsplit = p.nsplit;
  const int32_t* idx_row = p.idx + static_cast<int64_t>(t) * p.topk;
  const int32_t* phys_row = p.phys ? p.phys + static_cast<int64_t>(t) * p.topk : nullptr;
  if (tid == 0) {
    mbar_init(ready, THREADS);
    mbar_init(s_full, 1);
    mbar_init(p_full, 12);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abortf = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  // Everything above touches only this CTA; the selection comes from the kernel before.
  grid_dep_wait();
  grid_dep_launch();

  // ---- selected entries of this split -> byte offsets of their latent records
  const int e0 = split * kSelTile;
  if (tid < kSelTile) {
    const int e = e0 + tid;
    int64_t off = -1;
    const int sv = e < p.topk ? __ldcg((phys_row ? phys_row : idx_row) + e) : -1;
    if (sv >= 0) {
      int prow = -1;
      int slot = 0;
      bool present = true;
      if (phys_row) {
        prow = sv >> p.pool.log2_bs;
        slot = sv & (p.pool.bs - 1);
      } else {
        int req = __ldg(p.b.q_req + t);
        const int pos = __ldg(p.b.q_pos + t);
        if (req < 0 || req >= p.b.B) {
          atomicOr(p.status, DEV_BAD_BATCH);
          req = req < 0 ? 0 : p.b.B - 1;
        }
        const int64_t s_lim = static_cast<int64_t>(p.b.bt_stride) << p.pool.log2_bs;
        present = sv <= pos && sv < s_lim;
        if (present)
          prow = __ldg(p.b.bt + static_cast<int64_t>(req) * p.b.bt_stride + (sv >> p.pool.log2_bs));
        else
          atomicOr(p.status, DEV_BAD_BATCH);
        slot = sv & (p.pool.bs - 1);
      }
      if (present) {
        if (prow < 0 || prow >= p.pool.num_rows)
          atomicOr(p.status, DEV_BAD_BLOCK);
        else
          off = static_cast<int64_t>(prow) * p.pool.row_stride + p.pool.lat_off + static_cast<int64_t>(slot) * kLatDim;
      }
    }
    src_off[tid] = off;
    if (tid == 0) *has_work = sv >= 0;   // valid entries come first: the split has work iff its first is selected
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Abort ab{abortf, p.status};
  const bool work = *has_work != 0;

  if (work) {
    // ---- 1. gather: 128 records x 40 pieces of 16 B (pieces 36..39 repeat dims 512..575)
    const uint32_t lat_s = smem_u32(smem + OFF_LAT);
#pragma unroll 2
    for (int pc = tid; pc < kSelTile * 40; pc += THREADS) {
      const int tok = pc / 40, k = pc - tok * 40;
      const int64_t off = src_off[tok];
      const int c = k < 32 ? (k >> 3) : 4;
      const int ci = k < 32 ? (k & 7) : (k - 32);
      const int sb = k < 36 ? k : k - 4;
      const uint8_t* src = p.pool.pool + (off >= 0 ? off + 16 * sb : 0);
      const uint32_t dst = lat_s + c * LCHUNK + tok * 128 + ((ci ^ (tok & 7)) << 4);
      cp_async16(dst, src, off >= 0 ? 16u : 0u);
    }
    // ---- 2. query terms (12 warps x 8 heads; 4 lanes per head, 144 dims each)
    if (warp < 12) {
      const int h = warp * 8 + (lane >> 2), m = lane & 3;
      const uint4* qsrc = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(t) * kMlaHeads + h) * kLatDim +
                                                         144 * m);
      // pass 1: the head's largest |q| (18 loads in flight); pass 2 reloads from L1
      float amax = 0.f;
      {
        uint4 v[18];
#pragma unroll
        for (int i = 0; i < 18; ++i) v[i] = __ldg(qsrc + i);
#pragma unroll
        for (int i = 0; i < 18; ++i) {
          const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] << 16)));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] & 0xFFFF0000u)));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int k2 = q_scale_log2(amax);
      const float sc = __uint_as_float(static_cast<uint32_t>(k2 + 127) << 23);
      if (m == 0) qexp[h] = k2;
      uint8_t* qrow = smem + OFF_Q + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll 3
      for (int g = 0; g < 9; ++g) {        // 16 dims per group: loads 2g, 2g + 1
        const int G = 9 * m + g;           // global 16-dim group, 0..35
        uint32_t hi[4], lo[4];
        const uint4 xv[2] = {__ldg(qsrc + 2 * g), __ldg(qsrc + 2 * g + 1)};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint4 x = xv[half];
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int j = 0; j < 2; ++j) {     // 4 values -> 4 bytes of each term
            const float a0 = __uint_as_float(w4[2 * j] << 16) * sc;
            const float a1 = __uint_as_float(w4[2 * j] & 0xFFFF0000u) * sc;
            const float a2 = __uint_as_float(w4[2 * j + 1] << 16) * sc;
            const float a3 = __uint_as_float(w4[2 * j + 1] & 0xFFFF0000u) * sc;
            const uint32_t h01 = f2_to_e4m3x2(a0, a1), h23 = f2_to_e4m3x2(a2, a3);
            const float2 b01 = e4m3x2_to_f2(h01), b23 = e4m3x2_to_f2(h23);
            const uint32_t l01 = f2_to_e4m3x2(a0 - b01.x, a1 - b01.y), l23 = f2_to_e4m3x2(a2 - b23.x, a3 - b23.y);
            hi[2 * half + j] = h01 | (h23 << 16);
            lo[2 * half + j] = l01 | (l23 << 16);
          }
        }
        const int hc = G < 32 ? (G >> 3) : 4, hi_i = G < 32 ? (G & 7) : (G - 32);
        const int lc = G < 32 ? 5 + (G >> 3) : 4, lo_i = G < 32 ? (G & 7) : (G - 28);
        *reinterpret_cast<uint4*>(qrow + hc * QCHUNK + ((hi_i ^ (h & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(qrow + lc * QCHUNK + ((lo_i ^ (h & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();   // the copies and the query terms are read by the tensor core
    mbar_arrive(ready);

    if (warp == MMA_WARP && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_qk = make_idesc(0, 0, false, false, 128, 128);
      const uint32_t idesc_pv = make_idesc(0, 0, true, false, 128, kMlaHeads);
      const uint64_t dq = make_sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);       // query terms, K-major
      const uint64_t dl = make_sdesc_sw128(smem_u32(smem + OFF_LAT), 16, 1024);     // latents, K-major (QK)
      const uint64_t dv = make_sdesc_sw128(smem_u32(smem + OFF_LAT), LCHUNK, 1024); // latents, MN-major (PV)
      const uint64_t dp = make_sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);       // P terms, K-major
      bool ok = mbar_wait(ready, 0, ab);
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < NQCHUNK; ++i) {
          const int lc = i < 4 ? i : (i == 4 ? 4 : i - 5);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8f6f4(tmem + S_COL, dq + ((i * QCHUNK + 32 * kk) >> 4), dl + ((lc * LCHUNK + 32 * kk) >> 4),
                       idesc_qk, (i | kk) ? 1u : 0u);
        }
        tc_commit(s_full);
        ok = mbar_wait(p_full, 0, ab);
      }
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int vb = 0; vb < 4; ++vb)
#pragma unroll 1
          for (int tm = 0; tm < 3; ++tm)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8f6f4(tmem + O_COL + 96 * vb, dv + ((vb * LCHUNK + kk * 4096) >> 4),
                         dp + ((tm * P_TERM + 32 * kk) >> 4), idesc_pv, (tm | kk) ? 1u : 0u);
        tc_commit(o_done);
      } else {
        tc_commit(drain);
        drain_wait(drain, 0);
      }
    } else if ((warp & 3) != 3) {
      // -------------------------------------- softmax: 12 warps, 4 per head quarter
      const int quarter = warp & 3, u = warp >> 2;   // heads 32 quarter.., tokens 32 u ..
      const int h = quarter * 32 + lane;
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      if (__all_sync(0xffffffffu, mbar_wait(s_full, 0, ab))) {   // uniform over the warp (aligned loads below)
        tc_fence_after();
        uint32_t rr[32];
        DSA_TMEM_LD32(tmem + S_COL + 32 * u + lane_off, rr);
        tmem_wait_ld();
        const float c = p.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 - qexp[h]) << 23);
        float* x = reinterpret_cast<float*>(rr);   // logits in log2 units, in place
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const bool valid = src_off[32 * u + j] >= 0;
          x[j] = valid ? __uint_as_float(rr[j]) * c : -INFINITY;
          mx = fmaxf(mx, x[j]);
        }
        red_m[u * 96 + h] = mx;
        named_bar_sync(1, 384);
        const float m = fmaxf(fmaxf(red_m[h], red_m[96 + h]), fmaxf(red_m[192 + h], red_m[288 + h]));
        const float base = m == -INFINITY ? 0.f : 8.f - m;   // p' = 2^(x - m + 8) <= 256 (0 for absent tokens)
        float l = 0.f;
        uint32_t t0[8], t1[8], t2[8];   // the three e4m3 terms of 32 values, 4 per word
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float p0 = ex2_approx(x[2 * j] + base), p1 = ex2_approx(x[2 * j + 1] + base);
          const __half2 ph = __floats2half2_rn(p0, p1);
          const float2 pf = __half22float2(ph);
          l += pf.x + pf.y;
          const uint32_t a = h2_to_e4m3x2(ph);
          const __half2 r1 = __hsub2(ph, e4m3x2_to_h2(a));
          const uint32_t b = h2_to_e4m3x2(r1);
          const __half2 r2 = __hsub2(r1, e4m3x2_to_h2(b));
          const uint32_t cc = h2_to_e4m3x2(r2);
          const int w = j >> 1, sh = (j & 1) * 16;
          if (sh == 0) {
            t0[w] = a;
            t1[w] = b;
            t2[w] = cc;
          } else {
            t0[w] |= a << 16;
            t1[w] |= b << 16;
            t2[w] |= cc << 16;
          }
        }
        red_l[u * 96 + h] = l;
        uint8_t* prow = smem + OFF_Q + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int ch = ((2 * u + i) ^ (h & 7)) << 4;
          *reinterpret_cast<uint4*>(prow + ch) = make_uint4(t0[4 * i], t0[4 * i + 1], t0[4 * i + 2], t0[4 * i + 3]);
          *reinterpret_cast<uint4*>(prow + P_TERM + ch) =
              make_uint4(t1[4 * i], t1[4 * i + 1], t1[4 * i + 2], t1[4 * i + 3]);
          *reinterpret_cast<uint4*>(prow + 2 * P_TERM + ch) =
              make_uint4(t2[4 * i], t2[4 * i + 1], t2[4 * i + 2], t2[4 * i + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
      } else {
        named_bar_sync(1, 384);   // keep the softmax barrier's count whole
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
  }

  // ---- epilogue (all 16 warps)
  if (work) mbar_wait(o_done, 0, ab);
  __syncthreads();
  const bool good = work && !*reinterpret_cast<volatile int*>(abortf);
  if (tid < kMlaHeads) {   // this CTA's per-head (max, sum) in log2 units of p' = 2^(logit2 - max + 8)
    float m = -INFINITY, l = 0.f;
    if (good) {
      m = fmaxf(fmaxf(red_m[tid], red_m[96 + tid]), fmaxf(red_m[192 + tid], red_m[288 + tid]));
      l = (red_l[tid] + red_l[96 + tid]) + (red_l[192 + tid] + red_l[288 + tid]);
    }
    ml[tid] = make_float2(m, l);
    inv_l[tid] = l > 0.f ? 1.f / l : 0.f;
  }
  __syncthreads();
  __syncwarp();   // warp MMA_WARP comes from a divergent branch; the TMEM loads below are warp-collective
  tc_fence_after();
  const int quarter = warp & 3, vb = warp >> 2;   // TMEM lanes = dims 128 vb + 32 quarter + lane
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const int dim = vb * 128 + quarter * 32 + lane;
  if (nsplit == 1) {
    if (good) {
      uint16_t* stage = reinterpret_cast<uint16_t*>(smem + OFF_Q);   // [96 heads][512 dims] bf16
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {
        uint32_t rr[32];
        DSA_TMEM_LD32(tmem + O_COL + 96 * vb + 32 * c + lane_off, rr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(rr[i]) * inv_l[32 * c + i]);
          stage[(32 * c + i) * kVDim + dim] = *reinterpret_cast<const uint16_t*>(&bv);
        }
      }
      __syncthreads();
      uint4* gdst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(t) * kMlaHeads * kVDim);
      for (int i = tid; i < kMlaHeads * kVDim / 8; i += THREADS)
        gdst[i] = *reinterpret_cast<const uint4*>(stage + 8 * i);
      if (tid < kMlaHeads && p.lse)
        p.lse[static_cast<int64_t>(t) * kMlaHeads + tid] = (ml[tid].x - 8.f + log2f(ml[tid].y)) * 0.69314718055994531f;
    }
  } else {
    // normalised fp16 partial, [512 dims][96 heads] at a 208-byte pitch, in this CTA's shared memory
    if (good) {
      uint8_t* row = smem + OFF_Q + dim * STG_PITCH;
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {
        uint32_t rr[32];
        DSA_TMEM_LD32(tmem + O_COL + 96 * vb + 32 * c + lane_off, rr);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 8 * q + 2 * e;
            const __half2 hv = __floats2half2_rn(__uint_as_float(rr[i]) * inv_l[32 * c + i],
                                                 __uint_as_float(rr[i + 1]) * inv_l[32 * c + i + 1]);
            w4[e] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          *reinterpret_cast<uint4*>(row + 64 * c + 16 * q) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    }
    cluster_arrive();   // release: the partial and (max, sum) are visible to the cluster after the wait
    cluster_wait();
    // weights of every split for every head: w_j = 2^(m_j - M) l_j / L
    float* wgt = reinterpret_cast<float*>(smem + OFF_WGT);
    if (tid < kMlaHeads) {
      float2 v[MAX_SPLITS];
      float M = -INFINITY;
#pragma unroll
      for (int j = 0; j < MAX_SPLITS; ++j) {
        v[j] = make_float2(-INFINITY, 0.f);
        if (j < nsplit) {
          const uint32_t a = cluster_map(smem_u32(&ml[tid]), static_cast<uint32_t>(j));
          v[j].x = __uint_as_float(ld_cluster_u32(a));
          v[j].y = __uint_as_float(ld_cluster_u32(a + 4));
        }
        if (v[j].y > 0.f) M = fmaxf(M, v[j].x);
      }
      float L = 0.f;
#pragma unroll
      for (int j = 0; j < MAX_SPLITS; ++j) {
        const float w = v[j].y > 0.f ? exp2f(v[j].x - M) * v[j].y : 0.f;
        v[j].y = w;
        L += w;
      }
      const float inv = 1.f / L;
#pragma unroll
      for (int j = 0; j < MAX_SPLITS; ++j)
        if (j < nsplit) wgt[j * kMlaHeads + tid] = v[j].y * inv;
      if (split == 0 && p.lse)
        p.lse[static_cast<int64_t>(t) * kMlaHeads + tid] = (M - 8.f + log2f(L)) * 0.69314718055994531f;
    }
    __syncthreads();
    // the 32-dim blocks this CTA owns: sum over the cluster's partials, bf16 out
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem + OFF_TILE);   // [96 heads][32 dims]
    const int d = tid / 12, g = tid % 12;   // dim of the block, group of 8 heads (384 threads)
#pragma unroll 1
    for (int blk = split; blk < kVDim / 32; blk += nsplit) {
      if (tid < 384) {
        const uint32_t own = smem_u32(smem + OFF_Q + (blk * 32 + d) * STG_PITCH + 16 * g);
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int j0 = 0; j0 < MAX_SPLITS; j0 += MAX_SPLITS / 2) {   // eight splits' loads in flight at a time
          if (j0 >= nsplit) break;
          uint4 part[MAX_SPLITS / 2];
#pragma unroll
          for (int j = 0; j < MAX_SPLITS / 2; ++j)
            if (j0 + j < nsplit) part[j] = ld_cluster_v4(cluster_map(own, static_cast<uint32_t>(j0 + j)));
#pragma unroll
          for (int j = 0; j < MAX_SPLITS / 2; ++j) {
            if (j0 + j >= nsplit) break;
            const float4 wa = *reinterpret_cast<const float4*>(wgt + (j0 + j) * kMlaHeads + 8 * g);
            const float4 wb = *reinterpret_cast<const float4*>(wgt + (j0 + j) * kMlaHeads + 8 * g + 4);
            if (wa.x == 0.f && wa.y == 0.f && wa.z == 0.f && wa.w == 0.f && wb.x == 0.f && wb.y == 0.f &&
                wb.z == 0.f && wb.w == 0.f)
              continue;   // a split with nothing selected (its partial was never written)
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            const uint32_t w4[4] = {part[j].x, part[j].y, part[j].z, part[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
              acc[2 * e] = fmaf(wv[2 * e], f.x, acc[2 * e]);
              acc[2 * e + 1] = fmaf(wv[2 * e + 1], f.y, acc[2 * e + 1]);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) tile[(8 * g + e) * 32 + d] = __float2bfloat16_rn(acc[e]);
      }
      __syncthreads();
      if (tid < 384) {
        const int hh = tid >> 2, q = tid & 3;
        __nv_bfloat16* o = p.out + (static_cast<int64_t>(t) * kMlaHeads + hh) * kVDim + blk * 32 + 8 * q;
        *reinterpret_cast<uint4*>(o) = *reinterpret_cast<const uint4*>(tile + hh * 32 + 8 * q);
      }
      __syncthreads();
    }
    cluster_arrive_relaxed();   // done reading the other CTAs
    cluster_wait();             // and they are done reading this one
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Largest cluster of this kernel the device can hold at once (0: none), per context.
static int max_active_clusters(int csize) {
  static std::mutex mu;
  struct E {
    void* ctx;
    int csize, n;
  };
  static std::vector<E> cache;
  void* ctx = current_context();
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const E& e : cache)
      if (e.ctx == ctx && e.csize == csize) return e.n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize, 1);
  cfg.blockDim = dim3(mla8::THREADS);
  cfg.dynamicSmemBytes = mla8::SMEM_BYTES;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = csize;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, sparse_mla_fp8_kernel<0>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (ctx) cache.push_back({ctx, csize, n});
  return n;
}

bool sparse_mla_fp8_available(int nsplit) {
  if (nsplit < 1 || nsplit > mla8::MAX_SPLITS) return false;
  if (set_func_attr_once(reinterpret_cast<const void*>(sparse_mla_fp8_kernel<0>),
                         cudaFuncAttributeMaxDynamicSharedMemorySize, mla8::SMEM_BYTES) != cudaSuccess)
    return false;
  if (nsplit > 8 && set_func_attr_once(reinterpret_cast<const void*>(sparse_mla_fp8_kernel<0>),
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return false;
  return nsplit == 1 || max_active_clusters(nsplit) > 0;
}

cudaError_t launch_sparse_mla_fp8(const MlaParams& p, cudaStream_t st, bool chained) {
  if (p.b.T == 0) return cudaSuccess;
  return launch_ex(sparse_mla_fp8_kernel<0>, dim3(p.nsplit, p.b.T), dim3(mla8::THREADS), mla8::SMEM_BYTES, st,
                   chained, p.nsplit > 1 ? static_cast<unsigned>(p.nsplit) : 0u, p);
}

}  // namespace dsa

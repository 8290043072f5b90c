// mla_fp8.cu — sparse MLA over FP8 latents, the latents read once, straight into
// the tensor cores' operand tiles.
//
// vLLM K3.1 Pro day-0 post, "Sparse Attention in K3.1 Pro" (+ Figure 1): every
// query head attends exactly over only the selected tokens' 576-byte FP8
// latents ("KV cache footprint"); 96 absorbed query heads, value = first 512
// latent dims, NoPE ("What's new in Kimi K3.1 Pro").  Partial results of the
// splits of the selection are merged by log-sum-exp, as the post's DCP section
// merges partial outputs across GPUs ("Long context: decode context
// parallelism with a sparse indexer").
//
// One CTA per (query token, 128 selected tokens).  Per CTA:
//  1. Four threads per selected entry translate it to its latent record and
//     copy the 576 bytes with 16-byte cp.async directly into five
//     128-byte-swizzled K-chunks of [128 tokens x 128 B] (dims 0..511 in chunks
//     0..3; chunk 4 holds dims 512..575 twice).  No conversion: e4m3 is the
//     MMA's operand type.  The query arrives as two exact e4m3 terms per value
//     (mla_q.cuh), prepared once per token, with bulk copies.
//  2. S[head, token] = sum_k q_term[head, k] . latent[token, k] over the nine
//     query chunks: tcgen05.mma kind::f8f6f4, M = 128 (heads 0..95; lanes
//     96..127 are padding nobody reads), N = 128 tokens, K = 1152, fp32 in TMEM.
//     Heads on TMEM lanes make the softmax thread-local: four threads per head,
//     32 tokens each.
//  3. p = 2^(logit2 - max + 8) is rounded once to fp16 (11 significant bits),
//     then split exactly into three e4m3 terms (4 + 4 + 3 bits), written as
//     three K-major [96 heads x 128 tokens] operand tiles; the row sum is the
//     sum of the same fp16 values, so the normalisation matches the weights.
//  4. O^T[dim, head] += V^T[dim, token] . P^T[token, head] for the four 128-dim
//     blocks of the value, three terms each: M = 128 dims, N = 96 heads, K =
//     3 x 128; A is the gathered latent tile itself read MN-major (the same
//     bytes as step 2's B operand), B the P tiles.  TMEM: S in columns
//     [0, 128), O^T blocks at 128 + 96 v: 512 columns.
//  5. One split: O / l in bf16.  Several: the normalised fp16 partial and the
//     per-head (max, sum) go to the workspace, and the split combine of mla.cu
//     merges them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>
#include <vector>

#include "mla_q.cuh"
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
constexpr int OFF_ML = OFF_REDL + 4 * 96 * 4;     // [96] float2: this CTA's (max, sum)
constexpr int OFF_INV = OFF_ML + 96 * 8;          // [96] float: 1 / sum
constexpr int OFF_BARS = OFF_INV + 96 * 4;
constexpr int OFF_MISC = OFF_BARS + 8 * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
constexpr int P_TERM = 96 * 128;                  // one e4m3 term of P^T (12 KB), at OFF_Q
constexpr int MAX_SPLITS = 16;
constexpr int S_COL = 0;
constexpr int O_COL = 128;
constexpr int MMA_WARP = 3;                       // a warp of lane quarter 3, which has no softmax role
static_assert(OFF_LAT % 1024 == 0 && OFF_SMALL % 1024 == 0, "operand tiles are 1024-byte aligned");
static_assert(3 * P_TERM <= OFF_LAT, "P fits the query region");
static_assert(3 * kVDim * 64 <= OFF_LAT, "the staged fp16 partial fits the query region");
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

// pmap: the split partials [T * nsplit * 512 dim rows][96 heads] fp16, box 32 heads x 256
// rows, 64-byte swizzle (unused with one split).
template <int DUMMY>
__global__ void __launch_bounds__(mla8::THREADS, 1)
    sparse_mla_fp8_kernel(const __grid_constant__ CUtensorMap pmap, MlaParams p) {
  using namespace mla8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024_m8(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* s_full = bars + 1;   // QK done
  uint64_t* p_full = bars + 2;   // P written (12 softmax warps)
  uint64_t* o_done = bars + 3;   // PV done
  uint64_t* drain = bars + 4;
  uint64_t* q_full = bars + 5;   // the query terms and exponents are in shared memory (bulk copies)
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
  const int split = blockIdx.x;
  const int nsplit = p.nsplit;
  const int32_t* idx_row = p.idx + static_cast<int64_t>(t) * p.topk;
  const int32_t* phys_row = p.phys ? p.phys + static_cast<int64_t>(t) * p.topk : nullptr;
  if (tid == 0) {
    mbar_init(s_full, 1);
    mbar_init(p_full, 12);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(q_full, 1);
    *abortf = 0;
    fence_mbar_init();
    if (nsplit > 1) prefetch_tensormap(&pmap);   // a launch parameter: fetched before the wait
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  // Everything above touches only this CTA; the selection (and, in a layer step, the
  // query terms) come from the kernels before.
  grid_dep_wait();
  grid_dep_launch();
  if (tid == 0) {   // the token's query terms (issued by the thread that set up the barriers)
    const uint8_t* src = p.q_terms + static_cast<int64_t>(t) * kQTokenBytes;
    mbar_arrive_expect_tx(q_full, kQTokenBytes);
#pragma unroll 1
    for (int c = 0; c < kQChunks; ++c) bulk_load(smem + OFF_Q + c * QCHUNK, src + c * QCHUNK, QCHUNK, q_full);
    bulk_load(qexp, src + kQTermBytes, kMlaHeads * 4, q_full);
  }

  // ---- selection -> latent record -> gather.  Warp w takes the selected entries
  // (rows of the tile) w + 16 j, j < 8: lanes 0..7 translate them (lane j row w + 16 j),
  // then for each row all lanes copy its 576 bytes with 16-byte cp.async straight into
  // the operand tiles, 512 contiguous bytes per instruction: pieces 0..31 are dims
  // 0..511 (chunks 0..3), then lanes 0..3 copy dims 512..575 into chunk 4 and lanes
  // 4..7 the same dims again into chunk 4's upper half (the query's chunk 4 holds
  // hi | lo of those dims).
  {
    int64_t off = -1;
    int sv = -1;
    if (lane < 8) {
      const int rrow = warp + 16 * lane;
      const int e = split * kSelTile + rrow;
      sv = e < p.topk ? __ldcg((phys_row ? phys_row : idx_row) + e) : -1;
      if (sv >= 0) {
        int prow = -1;
        bool present = true;
        if (phys_row) {
          prow = sv >> p.pool.log2_bs;
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
        }
        if (present) {
          if (prow < 0 || prow >= p.pool.num_rows)
            atomicOr(p.status, DEV_BAD_BLOCK);
          else
            off = static_cast<int64_t>(prow) * p.pool.row_stride + p.pool.lat_off +
                  static_cast<int64_t>(sv & (p.pool.bs - 1)) * kLatDim;
        }
      }
      src_off[rrow] = off;
    }
    if (warp == 0 && lane == 0) *has_work = sv >= 0;   // valid entries come first: work iff the first is selected
    const uint32_t lat_s = smem_u32(smem + OFF_LAT);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t o = __shfl_sync(0xffffffffu, off, j);
      const int rrow = warp + 16 * j;
      const uint8_t* rec = p.pool.pool + (o >= 0 ? o : 0);
      const uint32_t nb = o >= 0 ? 16u : 0u;
      const uint32_t rb = lat_s + rrow * 128;
      const uint32_t sw = static_cast<uint32_t>(rrow & 7);
      cp_async16(rb + (lane >> 3) * LCHUNK + (((lane & 7) ^ sw) << 4), rec + 16 * lane, nb);
      if (lane < 8) cp_async16(rb + 4 * LCHUNK + ((lane ^ sw) << 4), rec + 512 + 16 * (lane & 3), nb);
    }
  }
  cp_async_wait_all();
  fence_proxy_async_smem();   // the copies are read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Abort ab{abortf, p.status};
  const bool work = *has_work != 0;

  if (work) {
    if (warp == MMA_WARP && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_qk = make_idesc(0, 0, false, false, 128, 128);
      const uint32_t idesc_pv = make_idesc(0, 0, true, false, 128, kMlaHeads);
      const uint64_t dq = make_sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);       // query terms, K-major
      const uint64_t dl = make_sdesc_sw128(smem_u32(smem + OFF_LAT), 16, 1024);     // latents, K-major (QK)
      const uint64_t dv = make_sdesc_sw128(smem_u32(smem + OFF_LAT), LCHUNK, 1024); // latents, MN-major (PV)
      const uint64_t dp = make_sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);       // P terms, K-major
      bool ok = mbar_wait(q_full, 0, ab);
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
      if (__all_sync(0xffffffffu, mbar_wait(s_full, 0, ab) && mbar_wait(q_full, 0, ab))) {   // uniform (aligned loads below)
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
  // 32 consecutive heads' reciprocal sums (8 vector loads)
  auto inv32 = [&](int c, float (&iv)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = *reinterpret_cast<const float4*>(inv_l + 32 * c + 4 * i);
      iv[4 * i] = x.x;
      iv[4 * i + 1] = x.y;
      iv[4 * i + 2] = x.z;
      iv[4 * i + 3] = x.w;
    }
  };
  if (nsplit == 1) {
    if (good) {
      uint16_t* stage = reinterpret_cast<uint16_t*>(smem + OFF_Q);   // [96 heads][512 dims] bf16
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {
        uint32_t rr[32];
        DSA_TMEM_LD32(tmem + O_COL + 96 * vb + 32 * c + lane_off, rr);
        float iv[32];
        inv32(c, iv);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(rr[i]) * iv[i]);
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
    // normalised fp16 partial [512 dims][96 heads] and (max - 8, sum) for the split
    // combine.  A split with nothing selected writes (-inf, 0) only.
    const int64_t ts = static_cast<int64_t>(t) * nsplit + split;
    if (good) {
      // Staged as three [512 dims x 32 heads] fp16 regions (64-byte rows, 64-byte
      // swizzle: 16-byte piece q of row r at q ^ ((r / 2) % 4), conflict-free), then
      // written by six tensor stores of 256 rows x 32 heads.
      auto stage32 = [&](const uint32_t (&rr)[32], int c) {
        float iv[32];
        inv32(c, iv);
        uint8_t* rowp = smem + OFF_Q + c * (kVDim * 64) + dim * 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w4[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int i = 8 * q + 2 * e2;
            const __half2 hv =
                __floats2half2_rn(__uint_as_float(rr[i]) * iv[i], __uint_as_float(rr[i + 1]) * iv[i + 1]);
            w4[e2] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          *reinterpret_cast<uint4*>(rowp + ((q ^ ((dim >> 1) & 3)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      };
      // each 32-head region leaves by its two tensor stores as soon as it is staged
      auto store32 = [&](int c) {
        fence_proxy_async_smem();   // the staged region is read by the tensor stores
        __syncthreads();
        if (tid == 0) {
#pragma unroll 1
          for (int hr = 0; hr < 2; ++hr)
            tma_store_2d(&pmap, smem + OFF_Q + c * (kVDim * 64) + hr * 256 * 64, 32 * c,
                         static_cast<int>(ts * kVDim) + 256 * hr);
          bulk_commit_group();
        }
      };
      uint32_t r0[32], r1[32];
      DSA_TMEM_LD32(tmem + O_COL + 96 * vb + lane_off, r0);   // two loads in flight, one wait
      DSA_TMEM_LD32(tmem + O_COL + 96 * vb + 32 + lane_off, r1);
      tmem_wait_ld();
      stage32(r0, 0);
      DSA_TMEM_LD32(tmem + O_COL + 96 * vb + 64 + lane_off, r0);
      store32(0);
      stage32(r1, 1);
      store32(1);
      tmem_wait_ld();
      stage32(r0, 2);
      store32(2);
      if (tid == 0) bulk_wait_group_read_all();   // the staging is read before the CTA's memory is released
    }
    if (tid < kMlaHeads) p.part_ml[ts * kMlaHeads + tid] = make_float2(ml[tid].x - 8.f, ml[tid].y);
  }
  if (tid == 0) drain_wait(q_full, 0);   // no copy into shared memory outlives the CTA
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// The query terms of every token (mla_q.cuh) for a standalone attention call: one
// warp per head, grid (T, 3) of 32 warps.
__global__ void __launch_bounds__(1024) mla_qprep_kernel(const __nv_bfloat16* q, uint8_t* terms) {
  const int t = blockIdx.x, h = blockIdx.y * 32 + (threadIdx.x >> 5);
  grid_dep_wait();
  uint8_t* tok = terms + static_cast<int64_t>(t) * kQTokenBytes;
  q_head_to_terms(q + static_cast<int64_t>(t) * kMlaHeads * kLatDim, h, tok, reinterpret_cast<int32_t*>(tok + kQTermBytes));
}

cudaError_t launch_mla_qprep(const __nv_bfloat16* q, uint8_t* terms, int T, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  return launch_ex(mla_qprep_kernel, dim3(T, 3), dim3(1024), 0, st, false, 0u, q, terms);
}

bool sparse_mla_fp8_available() {
  return set_func_attr_once(reinterpret_cast<const void*>(sparse_mla_fp8_kernel<0>),
                            cudaFuncAttributeMaxDynamicSharedMemorySize, mla8::SMEM_BYTES) == cudaSuccess;
}

// One CTA per (token, 128 selected tokens), then (several splits) the split combine.
cudaError_t launch_sparse_mla_fp8(const CUtensorMap& pmap, const CUtensorMap& cmap, const MlaParams& p, cudaStream_t st,
                                  bool chained) {
  if (p.b.T == 0) return cudaSuccess;
  const cudaError_t e = launch_ex(sparse_mla_fp8_kernel<0>, dim3(p.nsplit, p.b.T), dim3(mla8::THREADS),
                                  mla8::SMEM_BYTES, st, chained, 0u, pmap, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  return launch_mla_combine(cmap, p, st);
}

}  // namespace dsa

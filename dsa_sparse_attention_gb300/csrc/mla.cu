// mla.cu — sparse MLA over the selected latents on the 5th-generation tensor cores.
//
// vLLM K3.1 Pro day-0 post, "Sparse Attention in K3.1 Pro" (+ Figure 1): every
// query head attends exactly over only the selected tokens' latents (576-byte
// FP8, "KV cache footprint"); absorbed queries over 96 heads, the value is the
// first 512 latent dims ("What's new in Kimi K3.1 Pro": NoPE).  Partial outputs
// of several splits are combined by log-sum-exp, as the DCP section does across
// GPUs ("Long context: decode context parallelism with a sparse indexer").
//
// Design (one CTA per (query token, split of the selected list), 128 selected
// tokens per tile).  The contraction is written transposed so that 96 heads fill
// the MMA's N exactly and both accumulators fit TMEM:
//   S^T[token, head] = C[token, 0:576] . q[head, 0:576]      M=128, N=96, K=576  (bf16 x bf16)
//   O^T[dim, head]  += V^T[dim, token] . P^T[token, head]     M=128 (x4 dim blocks), N=96, K=128 (f16 x f16)
// TMEM: S^T in columns [0, 96), O^T blocks at 128 + 96 v (v = 0..3): 480 of 512.
// Softmax runs across TMEM lanes (tokens): per-head maxima with redux.sync.max.f32
// and a 4-warp exchange; the running maximum is only moved when a tile exceeds
// it by more than 2^8 (the output is unchanged: the final normalisation uses the
// same maximum), so O^T is rescaled in TMEM only on those rare tiles.
// Roles: warp 0 gathers the 128 selected latent rows of a tile with bulk copies
// (page translation per row) and streams q in 64-dim chunks with TMA; warp 1
// issues MMAs; warps 2..5 convert e4m3 -> bf16 (QK operand) and -> fp16 (PV
// operand) into 128-byte-swizzled tiles, run the softmax (P in fp16), and write
// the output (or the fp32 partial for the LSE combine).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "params.cuh"

namespace dsa {


namespace mla {
constexpr int RAW_STRIDE = 592;                   // 576 + 16: conflict-free row reads
constexpr int OFF_RAW = 0;
constexpr int RAW_BYTES = kSelTile * RAW_STRIDE;  // 75,776
constexpr int OFF_Q = 76800;                      // 2 x [96 x 128 B]
constexpr int Q_SLOT = kMlaHeads * 128;
constexpr int OFF_C = OFF_Q + 2 * Q_SLOT;         // 2 x [128 x 128 B]
constexpr int C_SLOT = kSelTile * 128;
constexpr int OFF_P = OFF_C + 2 * C_SLOT;         // P^T: 2 head atoms x 16 token groups x 1 KB
constexpr int P_BYTES = 2 * 16 * 1024;
constexpr int OFF_V = OFF_P + P_BYTES;            // 2 x [128 dims x 64 tokens] f16
constexpr int V_SLOT = 2 * 8 * 1024;
constexpr int OFF_RED = OFF_V + 2 * V_SLOT;       // 4 x 96 floats
constexpr int OFF_MUSE = OFF_RED + 4 * 96 * 4;    // 96 floats
constexpr int OFF_ALPHA = OFF_MUSE + 96 * 4;      // 96 floats
constexpr int OFF_LFIN = OFF_ALPHA + 96 * 4;      // 96 floats
constexpr int OFF_RED2 = OFF_LFIN + 96 * 4;       // 4 x 96 floats
constexpr int OFF_BARS = OFF_RED2 + 4 * 96 * 4;
constexpr int N_BARS = 16;
constexpr int OFF_MISC = OFF_BARS + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int S_COL = 0;
constexpr int O_COL = 128;
constexpr float TAU = 8.0f;                       // log2 headroom before the running max moves
static_assert(OFF_Q % 1024 == 0 && OFF_C % 1024 == 0 && OFF_P % 1024 == 0 && OFF_V % 1024 == 0, "align");
static_assert(OFF_Q >= RAW_BYTES, "raw");
static_assert(SMEM_BYTES <= 232448, "smem");
}  // namespace mla

__device__ __forceinline__ uint8_t* align1024_mla(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void drain_wait_mla(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(addr, parity))
    if (globaltimer() - t0 > 200000000ull) break;
}

// 16 e4m3 bytes -> 16 bf16 values (exact), packed as 8 x bf16x2.
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 in, uint32_t (&o)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
    const float2 flo = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 fhi = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    const __nv_bfloat162 blo = __floats2bfloat162_rn(flo.x, flo.y);
    const __nv_bfloat162 bhi = __floats2bfloat162_rn(fhi.x, fhi.y);
    o[2 * i] = *reinterpret_cast<const uint32_t*>(&blo);
    o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&bhi);
  }
}

// 16 e4m3 bytes -> 16 fp16 values (exact), packed as 8 x f16x2.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 in, uint32_t (&o)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
    o[2 * i] = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
    o[2 * i + 1] = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
  }
}

// Butterfly "transpose" reductions over a warp: on entry every lane holds 32
// values (one per head j); on exit lane l holds the reduction over all 32 lanes
// of head l.  31 shuffles per 32 heads.  `v` is destroyed.
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? v[j] : v[j + half];
      const float keep = upper ? v[j + half] : v[j];
      const float recv = __shfl_xor_sync(0xffffffffu, send, half);
      v[j] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

__device__ __forceinline__ void sts128(uint8_t* p, const uint32_t* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(v[0], v[1], v[2], v[3]);
}

__global__ void __launch_bounds__(mla::THREADS, 1)
    sparse_mla_fp8_kernel(const __grid_constant__ CUtensorMap qmap, MlaParams p) {
  using namespace mla;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024_mla(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* raw_full = bars + 0;
  uint64_t* raw_empty = bars + 1;
  uint64_t* q_full = bars + 2;    // [2]
  uint64_t* q_empty = bars + 4;   // [2]
  uint64_t* c_full = bars + 6;    // [2]
  uint64_t* c_empty = bars + 8;   // [2]
  uint64_t* v_full = bars + 10;   // [2]
  uint64_t* v_empty = bars + 12;  // [2]
  uint64_t* s_full = bars + 14;
  uint64_t* misc_bar = bars + 15;
  __shared__ __align__(8) uint64_t s_free, p_full, o_done, drain;
  __shared__ int n_valid_sh;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* abortf = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  float* red = reinterpret_cast<float*>(smem + OFF_RED);
  float* m_use = reinterpret_cast<float*>(smem + OFF_MUSE);
  float* alpha_sh = reinterpret_cast<float*>(smem + OFF_ALPHA);
  float* l_fin = reinterpret_cast<float*>(smem + OFF_LFIN);
  float* red2 = reinterpret_cast<float*>(smem + OFF_RED2);
  int* rescale_sh = reinterpret_cast<int*>(smem + OFF_MISC + 16);
  (void)misc_bar;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.y;
  const int split = blockIdx.x;
  int req, pos;
  load_token(p.b, t, p.status, req, pos);
  const int32_t* idx_row = p.idx + static_cast<int64_t>(t) * p.topk;

  if (threadIdx.x == 0) {
    mbar_init(raw_full, 1);
    mbar_init(raw_empty, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&c_full[i], 4);
      mbar_init(&c_empty[i], 1);
      mbar_init(&v_full[i], 4);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(&s_free, 4);
    mbar_init(&p_full, 4);
    mbar_init(&o_done, 1);
    mbar_init(&drain, 1);
    *abortf = 0;
    n_valid_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // number of valid (non-negative) selected entries; they come first
  {
    int cnt = 0;
    for (int i = threadIdx.x; i < p.topk; i += blockDim.x) cnt += idx_row[i] >= 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0 && cnt) atomicAdd(&n_valid_sh, cnt);
  }
  if (warp == 1) tmem_alloc(tslot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Abort ab{abortf, p.status};
  const int n_valid = n_valid_sh;
  const int n_tiles = static_cast<int>(cdiv(n_valid, kSelTile));
  const int j0 = split * p.tps;
  const int j1 = min(n_tiles, j0 + p.tps);
  const int64_t ts = static_cast<int64_t>(t) * p.nsplit + split;

  if (j0 >= j1) {
    // nothing selected for this split: an empty partial (weight 0 in the combine)
    if (p.nsplit > 1 && threadIdx.x < kMlaHeads) p.part_ml[ts * kMlaHeads + threadIdx.x] = make_float2(-INFINITY, 0.f);
  } else if (warp == 0) {
    // --------------------------------------------------------------- producer
    if (lane == 0) prefetch_tensormap(&qmap);
    const int32_t* btrow = p.b.bt + static_cast<int64_t>(req) * p.b.bt_stride;
    const int bsm = p.pool.bs - 1;
    int qc = 0;
    bool ok = true;
    int issued_tiles = 0;
    for (int j = j0; j < j1 && ok; ++j) {
      const int jt = j - j0;
      if (jt > 0 && !(ok = mbar_wait(raw_empty, (jt - 1) & 1, ab))) break;
      const uint8_t* src[4];
      uint32_t nrow = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        const int e = j * kSelTile + r;
        src[i] = nullptr;
        if (e < n_valid) {
          int s = idx_row[e];
          if (s < 0 || s > pos) {
            atomicOr(p.status, DEV_BAD_BATCH);
          } else {
            const int row = btrow[s >> p.pool.log2_bs];
            if (row < 0 || row >= p.pool.num_rows) {
              atomicOr(p.status, DEV_BAD_BLOCK);
            } else {
              src[i] = p.pool.pool + static_cast<int64_t>(row) * p.pool.row_stride + p.pool.lat_off +
                       static_cast<int64_t>(s & bsm) * kLatDim;
              ++nrow;
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) nrow += __shfl_xor_sync(0xffffffffu, nrow, o);
      if (lane == 0) mbar_arrive_expect_tx(raw_full, nrow * kLatDim);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (src[i]) bulk_load(smem + OFF_RAW + (lane + 32 * i) * RAW_STRIDE, src[i], kLatDim, raw_full);
      ++issued_tiles;
      // q in 9 chunks of 64 dims
      for (int kc = 0; kc < kLatDim / 64 && ok; ++kc, ++qc) {
        const int slot = qc & 1;
        if (qc >= 2) ok = mbar_wait(&q_empty[slot], ((qc >> 1) - 1) & 1, ab);
        if (ok && lane == 0) {
          mbar_arrive_expect_tx(&q_full[slot], Q_SLOT);
          tma_load_2d(smem + OFF_Q + slot * Q_SLOT, &qmap, &q_full[slot], kc * 64, t * kMlaHeads);
        }
        __syncwarp();
      }
    }
    if (!ok && issued_tiles > 0) drain_wait_mla(raw_full, (issued_tiles - 1) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(1, 1, false, false, 128, kMlaHeads);
      const uint32_t idesc_pv = make_idesc(0, 0, true, true, 128, kMlaHeads);
      int cc = 0, vc = 0;
      bool ok = true;
      for (int j = j0; j < j1 && ok; ++j) {
        const int jt = j - j0;
        if (jt > 0 && !(ok = mbar_wait(&s_free, (jt - 1) & 1, ab))) break;
        for (int kc = 0; kc < kLatDim / 64; ++kc, ++cc) {
          const int slot = cc & 1;
          const uint32_t ph = (cc >> 1) & 1;
          if (!(ok = mbar_wait(&c_full[slot], ph, ab))) break;
          if (!(ok = mbar_wait(&q_full[slot], ph, ab))) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + OFF_C + slot * C_SLOT);
          const uint32_t b0 = smem_u32(smem + OFF_Q + slot * Q_SLOT);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(tmem + S_COL, make_sdesc_sw128(a0 + 32 * kk, 16, 1024), make_sdesc_sw128(b0 + 32 * kk, 16, 1024),
                    idesc_qk, (kc | kk) ? 1u : 0u);
          tc_commit(&c_empty[slot]);
          tc_commit(&q_empty[slot]);
        }
        if (!ok) break;
        tc_commit(s_full);
        if (!(ok = mbar_wait(&p_full, jt & 1, ab))) break;
        tc_fence_after();
        for (int v = 0; v < 4 && ok; ++v) {
          for (int kh = 0; kh < 2; ++kh, ++vc) {
            const int slot = vc & 1;
            if (!(ok = mbar_wait(&v_full[slot], (vc >> 1) & 1, ab))) break;
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + OFF_V + slot * V_SLOT);
            const uint32_t b0 = smem_u32(smem + OFF_P);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f16(tmem + O_COL + 96 * v, make_sdesc_sw128(a0 + k * 2048, 8192, 1024),
                      make_sdesc_sw128(b0 + (kh * 8 + k * 2) * 1024, 16384, 1024), idesc_pv,
                      (jt > 0 || kh > 0 || k > 0) ? 1u : 0u);
            tc_commit(&v_empty[slot]);
          }
        }
        if (!ok) break;
        tc_commit(&o_done);
      }
      if (!ok) {
        tc_commit(&drain);
        drain_wait_mla(&drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------ math warps (2..5)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;          // token lane within the tile
    const int mt = threadIdx.x - 64;            // 0..127
    float m_run[3] = {-INFINITY, -INFINITY, -INFINITY};   // per head (lane + 32 i), log2 units
    float l_run[3] = {0.f, 0.f, 0.f};                      // warp 2 only: running sums
    float alpha_r[3] = {1.f, 1.f, 1.f};
    int cc = 0, vc = 0;
    bool ok = true;
    for (int j = j0; j < j1 && ok; ++j) {
      const int jt = j - j0;
      if (!(ok = mbar_wait(raw_full, jt & 1, ab))) break;
      const uint8_t* raw = smem + OFF_RAW;
      // validity of this thread's token row (the producer skipped invalid rows)
      bool valid = false;
      {
        const int e = j * kSelTile + r;
        if (e < n_valid) {
          const int s = idx_row[e];
          if (s >= 0 && s <= pos) {
            const int row = p.b.bt[static_cast<int64_t>(req) * p.b.bt_stride + (s >> p.pool.log2_bs)];
            valid = row >= 0 && row < p.pool.num_rows;
          }
        }
      }
      // ---- C chunks (bf16, K-major, 128-byte swizzle): thread r writes row r
      for (int kc = 0; kc < kLatDim / 64; ++kc, ++cc) {
        const int slot = cc & 1;
        if (cc >= 2 && !(ok = mbar_wait(&c_empty[slot], ((cc >> 1) - 1) & 1, ab))) break;
        uint8_t* dst = smem + OFF_C + slot * C_SLOT + (r >> 3) * 1024;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t o[8];
          if (valid) {
            const uint4 in = *reinterpret_cast<const uint4*>(raw + r * RAW_STRIDE + kc * 64 + q4 * 16);
            e4m3x16_to_bf16(in, o);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = 0;
          }
          sts128(dst + sw128_off(r & 7, 2 * q4), o);
          sts128(dst + sw128_off(r & 7, 2 * q4 + 1), o + 4);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c_full[slot]);
      }
      if (!ok) break;
      // ---- softmax over the tile's tokens (TMEM lanes) for each head (columns)
      if (!(ok = mbar_wait(s_full, jt & 1, ab))) break;
      tc_fence_after();
      float x[kMlaHeads];
      {
        uint32_t rr[32];
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          DSA_TMEM_LD32(tmem + S_COL + 32 * c + (static_cast<uint32_t>(quarter * 32) << 16), rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[32 * c + i] = valid ? __uint_as_float(rr[i]) * p.scale_log2 : -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free);
      // tile maxima per head: warp butterfly, then the 4 warps through shared memory
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        float tmp[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) tmp[i] = x[32 * c + i];
        red[quarter * kMlaHeads + 32 * c + lane] = warp_transpose_reduce32<true>(tmp);
      }
      named_bar_sync(1, 128);
      if (warp == 2) {
        bool moved = false;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const int h = lane + 32 * i;
          const float tm =
              fmaxf(fmaxf(red[h], red[kMlaHeads + h]), fmaxf(red[2 * kMlaHeads + h], red[3 * kMlaHeads + h]));
          const float mo = m_run[i];
          const float mn = (tm > mo + TAU) ? tm : mo;
          alpha_r[i] = (mn == mo) ? 1.f : exp2f(mo - mn);
          m_run[i] = mn;
          m_use[h] = mn;
          alpha_sh[h] = alpha_r[i];
          moved |= (mn != mo);
        }
        moved = __any_sync(0xffffffffu, moved);
        if (lane == 0) *rescale_sh = (moved && jt > 0) ? 1 : 0;
      }
      named_bar_sync(1, 128);
      const bool any_rescale = *reinterpret_cast<volatile int*>(rescale_sh) != 0;
      // PV of the previous tile must be done before P is overwritten or O rescaled
      if (jt > 0 && !(ok = mbar_wait(&o_done, (jt - 1) & 1, ab))) break;
      if (any_rescale) {
        tc_fence_after();
        for (int v = 0; v < 4; ++v) {
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            uint32_t rr[32];
            const uint32_t ta = tmem + O_COL + 96 * v + 32 * c + (static_cast<uint32_t>(quarter * 32) << 16);
            DSA_TMEM_LD32(ta, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha_sh[32 * c + i]);
            DSA_TMEM_ST32(ta, rr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
      }
      // P^T row r (fp16), MN-major: heads contiguous in 16-byte chunks of 8; row sums per head
      {
        uint8_t* prow = smem + OFF_P + (r >> 3) * 1024;
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          float pv[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pv[i] = valid ? exp2f(x[32 * c + i] - m_use[32 * c + i]) : 0.f;
#pragma unroll
          for (int cc4 = 0; cc4 < 4; ++cc4) {
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __half2 hp = __floats2half2_rn(pv[8 * cc4 + 2 * i], pv[8 * cc4 + 2 * i + 1]);
              o[i] = *reinterpret_cast<const uint32_t*>(&hp);
            }
            const int chunk = 4 * c + cc4;
            sts128(prow + (chunk >> 3) * 16384 + sw128_off(r & 7, chunk & 7), o);
          }
          red2[quarter * kMlaHeads + 32 * c + lane] = warp_transpose_reduce32<false>(pv);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
      named_bar_sync(1, 128);
      if (warp == 2) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const int h = lane + 32 * i;
          l_run[i] = l_run[i] * alpha_r[i] + red2[h] + red2[kMlaHeads + h] + red2[2 * kMlaHeads + h] +
                     red2[3 * kMlaHeads + h];
        }
      }
      // ---- V blocks (fp16, MN-major): block v = dims [128v, 128v+128), half kh = tokens [64kh, 64kh+64)
      for (int v = 0; v < 4 && ok; ++v) {
        for (int kh = 0; kh < 2; ++kh, ++vc) {
          const int slot = vc & 1;
          if (vc >= 2 && !(ok = mbar_wait(&v_empty[slot], ((vc >> 1) - 1) & 1, ab))) break;
          const int tl = mt >> 1;            // token within the half (0..63)
          const int d2 = mt & 1;             // which 64-dim atom of the block
          const int row = kh * 64 + tl;
          bool rv = false;
          {
            const int e = j * kSelTile + row;
            if (e < n_valid) {
              const int s = idx_row[e];
              if (s >= 0 && s <= pos) {
                const int prow = p.b.bt[static_cast<int64_t>(req) * p.b.bt_stride + (s >> p.pool.log2_bs)];
                rv = prow >= 0 && prow < p.pool.num_rows;
              }
            }
          }
          uint8_t* dst = smem + OFF_V + slot * V_SLOT + d2 * 8192 + (tl >> 3) * 1024;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t o[8];
            if (rv) {
              const uint4 in =
                  *reinterpret_cast<const uint4*>(raw + row * RAW_STRIDE + v * 128 + d2 * 64 + q4 * 16);
              e4m3x16_to_f16(in, o);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) o[i] = 0;
            }
            sts128(dst + sw128_off(tl & 7, 2 * q4), o);
            sts128(dst + sw128_off(tl & 7, 2 * q4 + 1), o + 4);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&v_full[slot]);
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(raw_empty);
    }
    // ---- epilogue: row sums across the 128 token lanes, then O / l or the partial
    if (ok) ok = mbar_wait(&o_done, (j1 - j0 - 1) & 1, ab);
    if (ok) {
      tc_fence_after();
      if (warp == 2) {
#pragma unroll
        for (int i = 0; i < 3; ++i) l_fin[lane + 32 * i] = l_run[i];
      }
      named_bar_sync(1, 128);
      if (p.nsplit == 1) {
        __nv_bfloat16* orow = p.out + static_cast<int64_t>(t) * kMlaHeads * kVDim;
        for (int v = 0; v < 4; ++v) {
          const int dim = v * 128 + r;
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            uint32_t rr[32];
            DSA_TMEM_LD32(tmem + O_COL + 96 * v + 32 * c + (static_cast<uint32_t>(quarter * 32) << 16), rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int h = 32 * c + i;
              orow[h * kVDim + dim] = __float2bfloat16_rn(__uint_as_float(rr[i]) / l_fin[h]);
            }
          }
        }
        if (p.lse && mt < kMlaHeads)
          p.lse[static_cast<int64_t>(t) * kMlaHeads + mt] = (m_use[mt] + log2f(l_fin[mt])) * 0.69314718055994531f;
      } else {
        float* po = p.part_o + ts * kMlaHeads * kVDim;
        for (int v = 0; v < 4; ++v) {
          const int dim = v * 128 + r;
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            uint32_t rr[32];
            DSA_TMEM_LD32(tmem + O_COL + 96 * v + 32 * c + (static_cast<uint32_t>(quarter * 32) << 16), rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) po[(32 * c + i) * kVDim + dim] = __uint_as_float(rr[i]);
          }
        }
        if (mt < kMlaHeads) p.part_ml[ts * kMlaHeads + mt] = make_float2(m_use[mt], l_fin[mt]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// Log-sum-exp combine of the split partials: grid (12, T), 256 threads = 8 heads x 32.
__global__ void __launch_bounds__(256) mla_combine_kernel(MlaParams p) {
  const int t = blockIdx.y;
  const int h = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t base = static_cast<int64_t>(t) * p.nsplit;
  float M = -INFINITY;
  for (int j = 0; j < p.nsplit; ++j) {
    const float2 ml = p.part_ml[(base + j) * kMlaHeads + h];
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float L = 0.f;
  for (int j = 0; j < p.nsplit; ++j) {
    const float2 ml = p.part_ml[(base + j) * kMlaHeads + h];
    if (!(ml.y > 0.f)) continue;
    const float wgt = exp2f(ml.x - M);
    L += wgt * ml.y;
    const float4* src = reinterpret_cast<const float4*>(p.part_o + ((base + j) * kMlaHeads + h) * kVDim);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldcg(src + lane + 32 * q);
      acc[4 * q + 0] = fmaf(wgt, v.x, acc[4 * q + 0]);
      acc[4 * q + 1] = fmaf(wgt, v.y, acc[4 * q + 1]);
      acc[4 * q + 2] = fmaf(wgt, v.z, acc[4 * q + 2]);
      acc[4 * q + 3] = fmaf(wgt, v.w, acc[4 * q + 3]);
    }
  }
  const float inv = 1.f / L;
  __nv_bfloat16* orow = p.out + (static_cast<int64_t>(t) * kMlaHeads + h) * kVDim;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[4 * q + 0] * inv, acc[4 * q + 1] * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[4 * q + 2] * inv, acc[4 * q + 3] * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(orow + 4 * (lane + 32 * q)) = u;
  }
  if (p.lse && lane == 0) p.lse[static_cast<int64_t>(t) * kMlaHeads + h] = (M + log2f(L)) * 0.69314718055994531f;
}

cudaError_t launch_sparse_mla(const CUtensorMap& qmap, const MlaParams& p, cudaStream_t st) {
  if (p.b.T == 0) return cudaSuccess;
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(sparse_mla_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  sparse_mla_fp8_kernel<<<dim3(p.nsplit, p.b.T), mla::THREADS, mla::SMEM_BYTES, st>>>(qmap, p);
  if (p.nsplit > 1) mla_combine_kernel<<<dim3(kMlaHeads / 8, p.b.T), 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa

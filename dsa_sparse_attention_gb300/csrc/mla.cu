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
// and a 4-warp exchange; per-head sums of P come from the tensor core (P^T
// against a block of ones, into the S columns once P is written); the running maximum is only moved when a tile exceeds
// it by more than 2^8 (the output is unchanged: the final normalisation uses the
// same maximum), so O^T is rescaled in TMEM only on those rare tiles.
// Roles: warp 0 loads the whole query (96 x 576 bf16) into shared memory with
// TMA before the kernel waits for the selection, so the load overlaps the
// kernel before it; warp 1 issues MMAs; warps 2..9 each own 16 selected rows of
// a tile: they translate each selection to its cache slot, load their half rows
// straight into registers, and convert them e4m3 (or NVFP4) -> bf16 (QK
// operand) and -> fp16 (PV operand) into 128-byte-swizzled tiles of a 4-slot
// ring; warps 10..13 run the softmax (P in fp16); all 12 math warps write the
// output (or the fp16 partial for the LSE combine).  On a CTA's last tile the
// second half of V lands in the query region (free once QK has completed), so
// all 32 PV MMAs issue after a single wait.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "params.cuh"

namespace dsa {


namespace mla {
constexpr int QCHUNKS = kLatDim / 64;             // 9 chunks of 64 dims
constexpr int Q_SLOT = kMlaHeads * 128;           // 12 KB: [96 heads x 128 B], 128-byte swizzle
constexpr int OFF_Q = 0;                          // the whole query; the output staging after the last MMA
constexpr int RSLOTS = 4;
constexpr int OFF_RING = QCHUNKS * Q_SLOT;        // RSLOTS x 16 KB: C chunks (QK) then V half-blocks (PV)
constexpr int RING_SLOT = 16384;
constexpr int OFF_P = OFF_RING + RSLOTS * RING_SLOT;   // P^T: 2 head atoms x 16 token groups x 1 KB
constexpr int P_BYTES = 2 * 16 * 1024;
constexpr int OFF_ONES = OFF_P + P_BYTES;         // one 8-row atom of fp16 ones (all rows of the sum operand)
constexpr int OFF_RED = OFF_ONES + 1024;          // 4 x 96 floats
constexpr int OFF_MUSE = OFF_RED + 4 * 96 * 4;    // 96 floats
constexpr int OFF_ALPHA = OFF_MUSE + 96 * 4;      // 96 floats
constexpr int OFF_LFIN = OFF_ALPHA + 96 * 4;      // 96 floats
constexpr int OFF_ROWOK = OFF_LFIN + 96 * 4;      // 2 x 128 bytes: selected row present (by tile parity)
constexpr int OFF_BARS = OFF_ROWOK + 256;
constexpr int N_BARS = 24;
constexpr int OFF_MISC = OFF_BARS + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
constexpr int THREADS = 448;                      // q loader, MMA, 8 converter warps, 4 softmax warps
// 14 warps put 4 on two of the SM's four register-file quarters (16K registers
// each): 128 registers per thread at most.
constexpr int CONV_WARPS = 8;
constexpr int SOFT_WARP0 = 2 + CONV_WARPS;        // first softmax warp
constexpr int TMEM_COLS = 512;
constexpr int S_COL = 0;
constexpr int O_COL = 128;
constexpr float TAU = 8.0f;                       // log2 headroom before the running max moves
static_assert(OFF_RING % 1024 == 0 && OFF_P % 1024 == 0 && OFF_ONES % 1024 == 0, "align");
static_assert(OFF_MUSE % 16 == 0 && OFF_ALPHA % 16 == 0, "per-head vectors are read 16 bytes at a time");
static_assert(kMlaHeads * kVDim * 2 <= OFF_RING && kVDim * 208 <= OFF_RING, "output staging fits the query region");
static_assert(4 * RING_SLOT <= OFF_RING, "four V half-blocks fit the query region");
static_assert(SMEM_BYTES <= 232448, "smem");
}  // namespace mla

__device__ __forceinline__ uint8_t* align1024_mla(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
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

// 16 NVFP4 values (8 packed bytes, element 2i in the low nibble of byte i) with
// their e4m3 block scale -> 16 fp16 values.  e2m1 x e4m3 has at most 6
// significant bits and lies in [2^-10, 2688]: exact in fp16 (and in bf16).
__device__ __forceinline__ void nvfp4x16_to_f16(const uint2 in, uint32_t scale_code, uint32_t (&o)[8]) {
  const __half sc = __half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(scale_code), __NV_E4M3));
  const __half2 sc2 = __half2(sc, sc);
  const uint32_t w[2] = {in.x, in.y};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>((w[i >> 2] >> (8 * (i & 3))) & 0xFFu),
                                                     __NV_E2M1);
    const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&r), sc2);
    o[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

__device__ __forceinline__ void nvfp4x16_to_bf16(const uint2 in, uint32_t scale_code, uint32_t (&o)[8]) {
  nvfp4x16_to_f16(in, scale_code, o);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&o[i]));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// 2^x on the multi-function unit (relative error about 2^-22; subnormal results flush to 0).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One 64-dim chunk of a converter thread's half row: dims [64 kc + 32 hf, +32).
// FP8: 32 bytes in a, b.  NVFP4: 16 bytes of packed values in a, the two e4m3
// block scales in the low bytes of s.  An absent row reads as zeros.
struct LatPiece {
  uint4 a, b;
  uint32_t s;
};

template <bool NV>
__device__ __forceinline__ LatPiece load_piece(const uint8_t* src, int kc, int hf) {
  LatPiece r;
  r.a = r.b = make_uint4(0, 0, 0, 0);
  r.s = 0;
  if (src) {
    if (NV) {
      r.a = __ldg(reinterpret_cast<const uint4*>(src + 32 * kc + 16 * hf));
      r.s = __ldg(reinterpret_cast<const uint16_t*>(src + 288 + 4 * kc + 2 * hf));
    } else {
      r.a = __ldg(reinterpret_cast<const uint4*>(src + 64 * kc + 32 * hf));
      r.b = __ldg(reinterpret_cast<const uint4*>(src + 64 * kc + 32 * hf + 16));
    }
  }
  return r;
}

// 16 values (piece q2 of the chunk) -> 8 packed bf16x2 / f16x2 words.
template <bool NV>
__device__ __forceinline__ void piece_to_bf16(const LatPiece& c, int q2, uint32_t (&o)[8]) {
  if (NV)
    nvfp4x16_to_bf16(q2 ? make_uint2(c.a.z, c.a.w) : make_uint2(c.a.x, c.a.y), (c.s >> (8 * q2)) & 0xFFu, o);
  else
    e4m3x16_to_bf16(q2 ? c.b : c.a, o);
}
template <bool NV>
__device__ __forceinline__ void piece_to_f16(const LatPiece& c, int q2, uint32_t (&o)[8]) {
  if (NV)
    nvfp4x16_to_f16(q2 ? make_uint2(c.a.z, c.a.w) : make_uint2(c.a.x, c.a.y), (c.s >> (8 * q2)) & 0xFFu, o);
  else
    e4m3x16_to_f16(q2 ? c.b : c.a, o);
}

// 32 consecutive floats of shared memory (16-byte aligned) through 8 vector loads.
__device__ __forceinline__ void lds_f32x32(const float* src, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 x = reinterpret_cast<const float4*>(src)[i];
    v[4 * i] = x.x;
    v[4 * i + 1] = x.y;
    v[4 * i + 2] = x.z;
    v[4 * i + 3] = x.w;
  }
}

__device__ __forceinline__ void sts128(uint8_t* p, const uint32_t* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(v[0], v[1], v[2], v[3]);
}

template <int LATF>
__global__ void __launch_bounds__(mla::THREADS, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap qmap, MlaParams p) {
  using namespace mla;
  constexpr bool NV = LATF == 1;
  constexpr int ROWB = NV ? 352 : kLatDim;             // bytes per latent record
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024_mla(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* q_full = bars + 0;
  uint64_t* rows_ready = bars + 1;
  uint64_t* ring_full = bars + 2;   // [RSLOTS]
  uint64_t* ring_empty = bars + 6;  // [RSLOTS]
  uint64_t* s_full = bars + 10;
  uint64_t* s_free = bars + 11;
  uint64_t* p_full = bars + 12;
  uint64_t* o_done = bars + 13;
  uint64_t* drain = bars + 14;
  uint64_t* sum_done = bars + 15;
  uint64_t* v_all = bars + 16;      // last tile: every V half-block is in shared memory (one arrival per converter warp)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* abortf = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  int* rescale_sh = reinterpret_cast<int*>(smem + OFF_MISC + 16);
  float* red = reinterpret_cast<float*>(smem + OFF_RED);
  float* m_use = reinterpret_cast<float*>(smem + OFF_MUSE);
  float* alpha_sh = reinterpret_cast<float*>(smem + OFF_ALPHA);
  float* l_fin = reinterpret_cast<float*>(smem + OFF_LFIN);
  uint8_t* rowok = smem + OFF_ROWOK;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.y;
  const int split = blockIdx.x;
  const int32_t* idx_row = p.idx + static_cast<int64_t>(t) * p.topk;
  const int32_t* phys_row = p.phys ? p.phys + static_cast<int64_t>(t) * p.topk : nullptr;
  const int32_t* sel_row = phys_row ? phys_row : idx_row;   // both use -1 padding
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(rows_ready, CONV_WARPS);
    for (int i = 0; i < RSLOTS; ++i) {
      mbar_init(&ring_full[i], CONV_WARPS);
      mbar_init(&ring_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(sum_done, 1);
    mbar_init(v_all, CONV_WARPS);
    *abortf = 0;
    fence_mbar_init();
    // the query is an input of the call, not of the kernel before: load it now
    prefetch_tensormap(&qmap);
    mbar_arrive_expect_tx(q_full, QCHUNKS * Q_SLOT);
    #pragma unroll 1
    for (int kc = 0; kc < QCHUNKS; ++kc)
      tma_load_2d(smem + OFF_Q + kc * Q_SLOT, &qmap, q_full, kc * 64, t * kMlaHeads);
  }
  for (int i = threadIdx.x; i < 256; i += THREADS) reinterpret_cast<uint32_t*>(smem + OFF_ONES)[i] = 0x3C003C00u;
  fence_proxy_async_smem();   // the ones are read by the tensor core
  if (warp == 1) tmem_alloc(tslot, TMEM_COLS);
  // The set-up above overlaps the end of the kernel that writes the selection.
  grid_dep_wait();
  grid_dep_launch();
  // Tiles of this split that hold selected entries (valid entries come first, so
  // a tile is used iff its first entry is valid); every thread reads the same few words.
  const int ntiles_max = static_cast<int>(cdiv(p.topk, kSelTile));
  const int j0 = split * p.tps;
  int j1 = j0;
  for (int j = j0; j < min(ntiles_max, j0 + p.tps); ++j)
    if (__ldcg(sel_row + j * kSelTile) >= 0) j1 = j + 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Abort ab{abortf, p.status};
  const int64_t ts = static_cast<int64_t>(t) * p.nsplit + split;

  if (j0 >= j1) {
    // nothing selected for this split: an empty partial (weight 0 in the combine)
    if (p.nsplit > 1 && threadIdx.x < kMlaHeads) p.part_ml[ts * kMlaHeads + threadIdx.x] = make_float2(-INFINITY, 0.f);
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(1, 1, false, false, 128, kMlaHeads);
      const uint32_t idesc_pv = make_idesc(0, 0, true, true, 128, kMlaHeads);
      const uint32_t idesc_sum = make_idesc(0, 0, false, true, 128, kMlaHeads);
      // Descriptors of the first slot of each operand, built once; a byte offset X
      // moves the start-address field (16-byte units, no carry below 256 KB) by X >> 4.
      const uint64_t d_c = make_sdesc_sw128(smem_u32(smem + OFF_RING), 16, 1024);      // C chunk, K-major
      const uint64_t d_q = make_sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);         // q chunk, K-major
      const uint64_t d_vr = make_sdesc_sw128(smem_u32(smem + OFF_RING), 8192, 1024);   // V^T in the ring, MN-major
      const uint64_t d_vq = make_sdesc_sw128(smem_u32(smem + OFF_Q), 8192, 1024);      // V^T in the query region
      const uint64_t d_p = make_sdesc_sw128(smem_u32(smem + OFF_P), 16384, 1024);      // P^T, MN-major
      const uint64_t d_one = make_sdesc_sw128(smem_u32(smem + OFF_ONES), 16, 0);       // the ones atom, repeated
      constexpr uint64_t kSlot = RING_SLOT >> 4;
      int fc = 0;
      bool ok = mbar_wait(q_full, 0, ab);
      for (int j = j0; j < j1 && ok; ++j) {
        const int jt = j - j0;
        if (jt > 0 && !(ok = mbar_wait(s_free, (jt - 1) & 1, ab))) break;
#pragma unroll 1
        for (int kc = 0; kc < QCHUNKS; ++kc, ++fc) {
          const int slot = fc % RSLOTS;
          if (!(ok = mbar_wait_inline(&ring_full[slot], (fc / RSLOTS) & 1, ab))) break;
          tc_fence_after();
          const uint64_t a = d_c + slot * kSlot;
          const uint64_t b = d_q + kc * (Q_SLOT >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_f16(tmem + S_COL, a + 2 * kk, b + 2 * kk, idesc_qk, (kc | kk) ? 1u : 0u);
          tc_commit(&ring_empty[slot]);
        }
        if (!ok) break;
        tc_commit(s_full);
        if (!(ok = mbar_wait(p_full, jt & 1, ab))) break;
        tc_fence_after();
        // per-head sums of P: ones[128 x 128] . P^T into the S columns (every lane gets the sums);
        // the ones operand is one atom repeated (8-row-group stride 0, same 32-byte K step)
#pragma unroll
        for (int kh = 0; kh < 2; ++kh)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16(tmem + S_COL, d_one + 2 * k, d_p + (kh * 8 + k * 2) * 64, idesc_sum, (kh | k) ? 1u : 0u);
        tc_commit(sum_done);
        // PV.  On the CTA's last tile, half-blocks 0..3 sit in the next four ring slots
        // and 4..7 in the query region (free once QK is done): one wait covers all
        // eight and the 32 MMAs issue back to back (each wait, fence and commit costs
        // the issuing thread about as much as an MMA).  Earlier tiles go through the
        // ring, which the next tile's chunks reuse.
        const bool last = j == j1 - 1;
        if (last) {
          if (!(ok = mbar_wait_inline(v_all, 0, ab))) break;
          tc_fence_after();
#pragma unroll 1
          for (int v = 0; v < 4; ++v) {
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {
              const int f = 2 * v + kh;
              const uint64_t a = f < 4 ? d_vr + ((fc + f) % RSLOTS) * kSlot : d_vq + (f - 4) * kSlot;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16(tmem + O_COL + 96 * v, a + 128 * k, d_p + (kh * 8 + k * 2) * 64, idesc_pv,
                        (jt > 0 || kh > 0 || k > 0) ? 1u : 0u);
            }
          }
          fc += 4;   // the ring slots are not handed back: no chunk follows on this CTA
        } else {
#pragma unroll 1
          for (int v = 0; v < 4 && ok; ++v) {
#pragma unroll 1
            for (int kh = 0; kh < 2; ++kh) {
              if (!(ok = mbar_wait_inline(&ring_full[fc % RSLOTS], (fc / RSLOTS) & 1, ab))) break;
              const uint64_t a = d_vr + (fc % RSLOTS) * kSlot;
              tc_fence_after();
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16(tmem + O_COL + 96 * v, a + 128 * k, d_p + (kh * 8 + k * 2) * 64, idesc_pv,
                        (jt > 0 || kh > 0 || k > 0) ? 1u : 0u);
              tc_commit(&ring_empty[fc % RSLOTS]);
              ++fc;
            }
          }
          if (!ok) break;
        }
        tc_commit(o_done);
      }
      if (!ok) {
        tc_commit(drain);
        drain_wait(drain, 0);
      }
    }
  } else if (warp >= 2 && warp < SOFT_WARP0) {
    // ----------------------------------------------------- converters (2..9)
    const int ct = threadIdx.x - 64;            // 0..255
    const int row = ct >> 1, hf = ct & 1;       // this thread's half row: dims [64 kc + 32 hf, +32) of each chunk kc
    const int vg = (ct >> 5) >> 2;              // V half-block of this warp's rows: tokens [64 vg, +64)
    const int tl = row & 63;
    const int bsm = p.pool.bs - 1;
    int pos = 0;
    int64_t s_lim = 0;
    const int32_t* btrow = nullptr;
    if (!phys_row) {   // logical positions: translate through the block table
      int req = __ldg(p.b.q_req + t);
      pos = __ldg(p.b.q_pos + t);
      if (req < 0 || req >= p.b.B) {
        if (ct == 0) atomicOr(p.status, DEV_BAD_BATCH);
        req = req < 0 ? 0 : p.b.B - 1;
      }
      s_lim = static_cast<int64_t>(p.b.bt_stride) << p.pool.log2_bs;   // positions the table covers
      btrow = p.b.bt + static_cast<int64_t>(req) * p.b.bt_stride;
    }
    int fc = 0;
    bool ok = true;
    for (int j = j0; j < j1 && ok; ++j) {
      const int jt = j - j0;
      // selected entry -> latent record
      const int e = j * kSelTile + row;
      const int sv = e < p.topk ? __ldcg(sel_row + e) : -1;
      const uint8_t* src = nullptr;
      if (sv >= 0) {
        int prow = -1;
        bool present = true;
        if (phys_row) {
          prow = sv >> p.pool.log2_bs;   // physical slot from the top-k: no block-table lookup
        } else {
          present = sv <= pos && sv < s_lim;
          if (present)
            prow = __ldg(btrow + (sv >> p.pool.log2_bs));
          else if (hf == 0)
            atomicOr(p.status, DEV_BAD_BATCH);
        }
        if (present) {
          if (prow < 0 || prow >= p.pool.num_rows) {
            if (hf == 0) atomicOr(p.status, DEV_BAD_BLOCK);
          } else {
            src = p.pool.pool + static_cast<int64_t>(prow) * p.pool.row_stride + p.pool.lat_off +
                  static_cast<int64_t>(sv & bsm) * ROWB;
          }
        }
      }
      // Chunks are loaded through a short register pipeline inside rolled loops: the
      // code runs once per tile, and unrolled it would be fetched cold every time.
      if (hf == 0) rowok[(jt & 1) * kSelTile + row] = src != nullptr;
      __syncwarp();
      if (lane == 0) mbar_arrive(rows_ready);
      // C chunks (bf16, K-major, 128-byte swizzle): 128 rows x 64 dims per ring slot.
      // Four chunks in flight; a slot is reloaded right after its chunk is used (a
      // register copy of a load still in flight would wait for it).
      LatPiece cb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) cb[u] = load_piece<NV>(src, u, hf);
#pragma unroll 1
      for (int kb = 0; kb < QCHUNKS && ok; kb += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int kc = kb + u;
          if (kc >= QCHUNKS) break;
          const int slot = fc % RSLOTS;
          if (fc >= RSLOTS && !(ok = mbar_wait_inline(&ring_empty[slot], ((fc / RSLOTS) - 1) & 1, ab))) break;
          uint8_t* dst = smem + OFF_RING + slot * RING_SLOT + (row >> 3) * 1024;
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int q4 = 2 * hf + q2;          // 16-dim piece of the chunk
            uint32_t o[8];
            piece_to_bf16<NV>(cb[u], q2, o);
            sts128(dst + sw128_off(row & 7, 2 * q4), o);
            sts128(dst + sw128_off(row & 7, 2 * q4 + 1), o + 4);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ring_full[slot]);
          ++fc;
          if (kc + 4 < QCHUNKS) cb[u] = load_piece<NV>(src, kc + 4, hf);
        }
      }
      if (!ok) break;
      // V half-blocks (fp16, MN-major): block v = dims [128v, +128), half vg = tokens [64vg, +64).
      // The warps of rows 0..63 fill the even ring fills, those of rows 64..127 the odd ones;
      // four warps complete a fill, each arriving twice.  Two blocks' chunks in flight.
      LatPiece vbuf[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        vbuf[u][0] = load_piece<NV>(src, 2 * u, hf);
        vbuf[u][1] = load_piece<NV>(src, 2 * u + 1, hf);
      }
      const bool last = j == j1 - 1;   // V half-blocks 4..7 go to the query region (see the MMA issuer)
#pragma unroll 1
      for (int vb2 = 0; vb2 < 4 && ok; vb2 += 2) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int v = vb2 + u;
          const int f = 2 * v + vg;
          const bool in_q = last && f >= 4;
          uint8_t* base;
          int slot = 0;
          if (in_q) {
            if (!(ok = mbar_wait_inline(s_full, jt & 1, ab))) break;   // QK done: the query is no longer read
            base = smem + OFF_Q + (f - 4) * RING_SLOT + (tl >> 3) * 1024;
          } else {
            const int myfc = fc + f;
            slot = myfc % RSLOTS;
            if (myfc >= RSLOTS && !(ok = mbar_wait_inline(&ring_empty[slot], ((myfc / RSLOTS) - 1) & 1, ab))) break;
            base = smem + OFF_RING + slot * RING_SLOT + (tl >> 3) * 1024;
          }
#pragma unroll
          for (int a = 0; a < 2; ++a) {          // 64-dim atom a = chunk 2v + a
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              const int q4 = 2 * hf + q2;        // 16-dim piece within the atom
              uint32_t o[8];
              piece_to_f16<NV>(vbuf[u][a], q2, o);
              sts128(base + a * 8192 + sw128_off(tl & 7, 2 * q4), o);
              sts128(base + a * 8192 + sw128_off(tl & 7, 2 * q4 + 1), o + 4);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && !last) mbar_arrive_cnt(&ring_full[slot], 2);
          if (v + 2 < 4) {
            vbuf[u][0] = load_piece<NV>(src, 2 * v + 4, hf);
            vbuf[u][1] = load_piece<NV>(src, 2 * v + 5, hf);
          }
        }
      }
      if (!ok) break;
      if (last && lane == 0) mbar_arrive(v_all);   // after this warp's four fills (each fenced above)
      fc += last ? 4 : 8;
    }
  } else if (warp >= SOFT_WARP0) {
    // ---------------------------------------------- softmax warps (10..13)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;          // token lane within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float m_run[3] = {-INFINITY, -INFINITY, -INFINITY};   // per head (lane + 32 i), log2 units
    float l_run[3] = {0.f, 0.f, 0.f};                      // first softmax warp only: running sums
    float alpha_r[3] = {1.f, 1.f, 1.f};
    bool ok = true;
    for (int j = j0; j < j1 && ok; ++j) {
      const int jt = j - j0;
      if (!(ok = mbar_wait(s_full, jt & 1, ab))) break;
      if (!(ok = mbar_wait(rows_ready, jt & 1, ab))) break;   // rowok of this tile
      tc_fence_after();
      const bool valid = rowok[(jt & 1) * kSelTile + r] != 0;
      // tile maxima per head: one warp reduction per head, then the 4 warps through shared memory
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {
        uint32_t rr[32];
        DSA_TMEM_LD32(tmem + S_COL + 32 * c + lane_off, rr);
        tmem_wait_ld();
        float mine = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float m = warp_max_f32(valid ? __uint_as_float(rr[i]) * p.scale_log2 : -INFINITY);
          if (lane == i) mine = m;
        }
        red[quarter * kMlaHeads + 32 * c + lane] = mine;
      }
      named_bar_sync(1, 128);
      if (warp == SOFT_WARP0) {
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
      if (jt > 0 && !(ok = mbar_wait(o_done, (jt - 1) & 1, ab))) break;
      if (any_rescale) {
        tc_fence_after();
#pragma unroll 1
        for (int v = 0; v < 4; ++v) {
#pragma unroll 1
          for (int c = 0; c < 3; ++c) {
            uint32_t rr[32];
            const uint32_t ta = tmem + O_COL + 96 * v + 32 * c + lane_off;
            DSA_TMEM_LD32(ta, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha_sh[32 * c + i]);
            DSA_TMEM_ST32(ta, rr);
          }
        }
        tmem_wait_st();
      }
      // P^T row r (fp16), MN-major: heads contiguous in 16-byte chunks of 8; row sums per head
      {
        uint8_t* prow = smem + OFF_P + (r >> 3) * 1024;
#pragma unroll 1
        for (int c = 0; c < 3; ++c) {
          uint32_t rr[32];
          DSA_TMEM_LD32(tmem + S_COL + 32 * c + lane_off, rr);
          tmem_wait_ld();
          float pv[32];
          lds_f32x32(m_use + 32 * c, pv);
#pragma unroll
          for (int i = 0; i < 32; ++i) pv[i] = valid ? ex2_fast(__uint_as_float(rr[i]) * p.scale_log2 - pv[i]) : 0.f;
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
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(p_full);
        if (warp != SOFT_WARP0) mbar_arrive(s_free);
      }
      if (warp == SOFT_WARP0) {
        // this tile's per-head sums, from the S columns; then S may be overwritten
        if (!(ok = mbar_wait(sum_done, jt & 1, ab))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          float ls = 0.f;
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t rr[8];
            DSA_TMEM_LD8(tmem + S_COL + 32 * c + 8 * q + lane_off, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (lane == 8 * q + i) ls = __uint_as_float(rr[i]);
          }
          l_run[c] = l_run[c] * alpha_r[c] + ls;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
      }
    }
    // row sums (and their reciprocals) for the shared epilogue below
    if (ok && warp == SOFT_WARP0) {
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        l_fin[lane + 32 * i] = l_run[i];
        alpha_sh[lane + 32 * i] = 1.f / l_run[i];   // reused: 1 / sum
      }
    }
  }
  // ---- epilogue (all 12 math warps): O / l, or the normalised fp16 partial and
  // (max, sum).  TMEM (thread = dim) -> shared [head][512 dims] -> 16-byte stores.
  if (j0 < j1 && warp >= 2) {
    const int mw = warp - 2;                        // 0..11
    const int quarter = warp & 3;
    const int which = mw >> 2;                      // 0..2: the three warps of this lane quarter
    const int et = threadIdx.x - 64;                // 0..383
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    mbar_wait(o_done, (j1 - j0 - 1) & 1, ab);
    named_bar_sync(2, 384);
    // a failed wait sets the CTA abort flag before this barrier, so the test is uniform
    if (!*reinterpret_cast<volatile int*>(abortf)) {
      tc_fence_after();
      if (p.nsplit == 1) {
        // final output [head][512 dims] in bf16: through shared memory for 16-byte stores
        uint16_t* stage = reinterpret_cast<uint16_t*>(smem + OFF_Q);   // the query is no longer read
#pragma unroll 1
        for (int pc = which; pc < 12; pc += 3) {       // (block v, head chunk c) pairs
          const int v = pc / 3, c = pc % 3;
          uint32_t rr[32];
          DSA_TMEM_LD32(tmem + O_COL + 96 * v + 32 * c + lane_off, rr);
          tmem_wait_ld();
          const int dim = v * 128 + quarter * 32 + lane;
          float al[32];
          lds_f32x32(alpha_sh + 32 * c, al);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(rr[i]) * al[i]);
            stage[(32 * c + i) * kVDim + dim] = *reinterpret_cast<const uint16_t*>(&bv);
          }
        }
        named_bar_sync(2, 384);
        uint16_t* gbase = reinterpret_cast<uint16_t*>(p.out + static_cast<int64_t>(t) * kMlaHeads * kVDim);
        for (int i = et; i < kMlaHeads * kVDim / 8; i += 384)
          *reinterpret_cast<uint4*>(gbase + 8 * i) = *reinterpret_cast<const uint4*>(stage + 8 * i);
        if (et < kMlaHeads && p.lse)
          p.lse[static_cast<int64_t>(t) * kMlaHeads + et] = (m_use[et] + log2f(l_fin[et])) * 0.69314718055994531f;
      } else {
        // normalised fp16 partial, dim-major [512 dims][96 heads]: each thread owns a dim and
        // packs pairs of heads; rows are staged at a 208-byte pitch (conflict-free 16-byte
        // stores), then copied out with coalesced 16-byte stores
        constexpr int PITCH = 208;
        uint8_t* stg = smem + OFF_Q;   // the query is no longer read
        // this warp's head chunk c = which for the four dim blocks, two blocks per TMEM wait
        const int c = which;
        float al[32];
        lds_f32x32(alpha_sh + 32 * c, al);
#pragma unroll 1
        for (int v2 = 0; v2 < 4; v2 += 2) {
          uint32_t rr[2][32];
          DSA_TMEM_LD32(tmem + O_COL + 96 * v2 + 32 * c + lane_off, rr[0]);
          DSA_TMEM_LD32(tmem + O_COL + 96 * (v2 + 1) + 32 * c + lane_off, rr[1]);
          tmem_wait_ld();
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            uint8_t* row = stg + ((v2 + b) * 128 + quarter * 32 + lane) * PITCH + 64 * c;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 8 * q + 2 * e;
                const __half2 hv =
                    __floats2half2_rn(__uint_as_float(rr[b][i]) * al[i], __uint_as_float(rr[b][i + 1]) * al[i + 1]);
                w4[e] = *reinterpret_cast<const uint32_t*>(&hv);
              }
              sts128(row + 16 * q, w4);
            }
          }
        }
        named_bar_sync(2, 384);
        uint4* gdst = reinterpret_cast<uint4*>(p.part_o + ts * kVDim * kMlaHeads);
#pragma unroll 4
        for (int i = et; i < kVDim * (kMlaHeads / 8); i += 384)
          gdst[i] = *reinterpret_cast<const uint4*>(stg + (i / 12) * PITCH + (i % 12) * 16);
        if (et < kMlaHeads) p.part_ml[ts * kMlaHeads + et] = make_float2(m_use[et], l_fin[et]);
      }
    }
  }
  if (threadIdx.x == 0) drain_wait(q_full, 0);   // no copy into shared memory outlives the CTA
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// Log-sum-exp combine of the split partials (each partial normalised by its
// own sum): out = sum_j w_j l_j o_j / sum_j w_j l_j, w_j = 2^(m_j - max m).
// Grid (512 / 32 dims, T), 12 warps.  The token's partials of the block's 32 dims
// come into shared memory by TMA, four splits per copy (boxes of 96 heads x 32
// dims x 4 splits, 192-byte rows; a box past the token's last split reads bytes
// that are not used), each on its own barrier so the sums start while later
// splits land; the nsplit x 96 (max, sum) pairs come by one bulk copy and
// threads 0..95 turn them into weights (one thread per head).  Warp w takes the
// 32 heads of quad w % 3 and the 8 dims of octet w / 3; lane = (dim, group of 8
// heads), so a warp's reads of one split hit every bank equally and its weights
// are four 32-byte rows.  Splits with nothing selected (sum 0) take no part in
// the sum.  The [96 heads x 32 dims] result is staged for row stores.
constexpr int kCombDims = 32;
constexpr int kCombThreads = 384;
constexpr int kMaxSplits = kMaxTopk / kSelTile;
constexpr int kCombBoxSplits = 4;                                   // splits per TMA copy
constexpr int kCombMaxBoxes = kMaxSplits / kCombBoxSplits;
constexpr int kCombSplitBytes = kCombDims * kMlaHeads * 2;          // 6144: one split's 32 dims x 96 heads
static_assert(kMaxSplits % kCombBoxSplits == 0, "whole boxes");
__global__ void __launch_bounds__(kCombThreads)
    mla_combine_kernel(const __grid_constant__ CUtensorMap cmap, MlaParams p) {
  extern __shared__ uint8_t csm_raw[];
  uint8_t* csm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(csm_raw) + 127) & ~uintptr_t(127));
  const int ns = p.nsplit;
  const int nbox = (ns + kCombBoxSplits - 1) / kCombBoxSplits;
  const float2* mls = reinterpret_cast<const float2*>(csm + nbox * kCombBoxSplits * kCombSplitBytes);   // [ns][96]
  __shared__ __align__(16) float wgt[kMaxSplits][kMlaHeads];   // normalised weight per split and head
  __shared__ __align__(16) __nv_bfloat16 tile[kMlaHeads][kCombDims];
  __shared__ uint32_t used_mask;   // bit j: split j holds selected tokens
  __shared__ __align__(8) uint64_t bars[kCombMaxBoxes + 1];   // one per box, then the (max, sum) pairs
  __shared__ int abortf;
  const int t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i <= kCombMaxBoxes; ++i) mbar_init(&bars[i], 1);
    abortf = 0;
    fence_mbar_init();
    prefetch_tensormap(&cmap);
  }
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();   // the next chained kernel (the next layer step's scorer) may be scheduled
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[kCombMaxBoxes], static_cast<uint32_t>(ns) * kMlaHeads * 8);
    bulk_load(const_cast<float2*>(mls), p.part_ml + static_cast<int64_t>(t) * ns * kMlaHeads,
              static_cast<uint32_t>(ns) * kMlaHeads * 8, &bars[kCombMaxBoxes]);
  } else if (threadIdx.x >= 32 && threadIdx.x < 32 + nbox) {   // one box per thread of warp 1
    const int bx = threadIdx.x - 32;
    mbar_arrive_expect_tx(&bars[bx], kCombBoxSplits * kCombSplitBytes);
    tma_load_3d(csm + bx * kCombBoxSplits * kCombSplitBytes, &cmap, &bars[bx], 0, blockIdx.x * kCombDims,
                t * ns + bx * kCombBoxSplits);
  }
  const Abort ab{&abortf, p.status};
  // Loops over the splits are unrolled to the maximum with the split count as a
  // predicate: their shared-memory loads then issue together.
  if (threadIdx.x < kMlaHeads && mbar_wait(&bars[kCombMaxBoxes], 0, ab)) {
    const int h = threadIdx.x;
    float2 ml[kMaxSplits];
#pragma unroll
    for (int j = 0; j < kMaxSplits; ++j) ml[j] = j < ns ? mls[j * kMlaHeads + h] : make_float2(0.f, 0.f);
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxSplits; ++j)
      if (ml[j].y > 0.f) M = fmaxf(M, ml[j].x);
    float w[kMaxSplits];
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxSplits; ++j) {
      w[j] = ml[j].y > 0.f ? exp2f(ml[j].x - M) * ml[j].y : 0.f;
      L += w[j];
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int j = 0; j < kMaxSplits; ++j)
      if (j < ns) wgt[j][h] = w[j] * inv;
    if (h == 0) {   // a split is empty for all heads or for none
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < kMaxSplits; ++j) m |= static_cast<uint32_t>(ml[j].y > 0.f) << j;
      used_mask = m;
    }
    if (p.lse && blockIdx.x == 0)
      p.lse[static_cast<int64_t>(t) * kMlaHeads + h] = (M + log2f(L)) * 0.69314718055994531f;
  }
  __syncthreads();   // the weights (or a timeout) are visible
  const int grp = 4 * (warp % 3) + (lane & 3);   // heads 8 grp .. 8 grp + 7
  const int dim = 8 * (warp / 3) + (lane >> 2);  // of the block's 32
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const uint32_t um = abortf ? 0u : used_mask;
  bool ok = true;
#pragma unroll
  for (int bx = 0; bx < kCombMaxBoxes; ++bx) {
    if (bx >= nbox || !ok) break;
    ok = mbar_wait(&bars[bx], 0, ab);
#pragma unroll
    for (int jj = 0; jj < kCombBoxSplits; ++jj) {
      const int j = bx * kCombBoxSplits + jj;
      // predicated loads (an unused split contributes zeros): no branch between them
      const bool use = ok && ((um >> j) & 1u);
      const uint8_t* src = csm + j * kCombSplitBytes + dim * (kMlaHeads * 2) + grp * 16;
      const uint4 u = use ? *reinterpret_cast<const uint4*>(src) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
      const float4 wa = use ? *reinterpret_cast<const float4*>(&wgt[j][8 * grp]) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 wb = use ? *reinterpret_cast<const float4*>(&wgt[j][8 * grp + 4]) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
        acc[2 * e] = fmaf(wv[2 * e], f.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(wv[2 * e + 1], f.y, acc[2 * e + 1]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) tile[8 * grp + i][dim] = __float2bfloat16_rn(acc[i]);
  __syncthreads();
  if (!abortf) {   // uniform: read after the barrier
    // 96 rows of 32 dims (64 bytes): 4 x 16-byte stores per row
    __nv_bfloat16* o = p.out + static_cast<int64_t>(t) * kMlaHeads * kVDim + blockIdx.x * kCombDims;
    const int h = threadIdx.x >> 2, q = threadIdx.x & 3;
    *reinterpret_cast<uint4*>(o + h * kVDim + 8 * q) = *reinterpret_cast<const uint4*>(&tile[h][8 * q]);
  }
  if (threadIdx.x >= 32 && threadIdx.x < 32 + nbox) drain_wait(&bars[threadIdx.x - 32], 0);   // no copy outlives the CTA
  if (threadIdx.x == 0) drain_wait(&bars[kCombMaxBoxes], 0);
}

cudaError_t launch_mla_combine(const CUtensorMap& cmap, const MlaParams& p, cudaStream_t st) {
  const int nbox = (p.nsplit + kCombBoxSplits - 1) / kCombBoxSplits;
  const int smem = nbox * kCombBoxSplits * kCombSplitBytes + p.nsplit * kMlaHeads * 8 + 128;
  cudaError_t e = set_func_attr_once(reinterpret_cast<const void*>(mla_combine_kernel),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSplits * (kCombSplitBytes + kMlaHeads * 8) + 128);
  if (e != cudaSuccess) return e;
  return launch_ex(mla_combine_kernel, dim3(kVDim / kCombDims, p.b.T), dim3(kCombThreads), smem, st, true, 0u, cmap,
                   p);
}

template <int LATF>
static cudaError_t launch_mla_fmt(const CUtensorMap& qmap, const MlaParams& p, cudaStream_t st, bool chained) {
  cudaError_t e = set_func_attr_once(reinterpret_cast<const void*>(sparse_mla_kernel<LATF>),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_ex(sparse_mla_kernel<LATF>, dim3(p.nsplit, p.b.T), dim3(mla::THREADS), mla::SMEM_BYTES, st, chained,
                   0u, qmap, p);
}

cudaError_t launch_sparse_mla(const CUtensorMap& qmap, const CUtensorMap& cmap, const MlaParams& p, cudaStream_t st,
                              bool chained) {
  if (p.b.T == 0) return cudaSuccess;
  cudaError_t e =
      p.pool.lat_fmt == 1 ? launch_mla_fmt<1>(qmap, p, st, chained) : launch_mla_fmt<0>(qmap, p, st, chained);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  return launch_mla_combine(cmap, p, st);
}

}  // namespace dsa

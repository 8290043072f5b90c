// params.cuh — kernel parameter blocks and launcher declarations.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace dsa {

struct IndexerParams {
  PoolView pool;
  BatchView b;
  const float* w;          // [T, 32]
  float* scores;           // [T, ld]
  int64_t ld;
  const PlanHeader* hdr;
  const ScoreGroup* groups;
  uint32_t* status;
};

struct TopkParams {
  BatchView b;
  const float* scores;
  int64_t ld;
  int k;
  int chunk;          // scores per CTA
  uint32_t* hist1;    // [T, 2048]
  uint32_t* hist2;    // [T, 2048]
  uint32_t* hist3;    // [T, 1024]
  uint32_t* counts;   // [T, nchunks, 2] (greater, equal)
  int nchunks;
  int32_t* idx;       // [T, k]
  int32_t* phys;      // [T, k] or null
  int log2_bs;
  uint32_t* status;
};

struct MlaParams {
  PoolView pool;
  BatchView b;
  const int32_t* idx;      // [T, topk]
  int topk;
  float scale_log2;        // sm_scale * log2(e)
  int tps;                 // tiles per split
  int nsplit;
  __nv_bfloat16* out;      // [T, 96, 512]       (nsplit == 1)
  float* lse;              // [T, 96] or null    (nsplit == 1)
  float* part_o;           // [T, nsplit, 96, 512] (nsplit > 1)
  float2* part_ml;         // [T, nsplit, 96]      (nsplit > 1): (max in log2 units, sum)
  uint32_t* status;
};

cudaError_t launch_plan_groups(const BatchView& b, int G, ScoreGroup* groups, PlanHeader* hdr, uint32_t* status,
                               cudaStream_t st);
cudaError_t launch_indexer_fp8(const CUtensorMap& kmap, const CUtensorMap& qmap, const IndexerParams& p, int G,
                               int grid, cudaStream_t st);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t st);
cudaError_t launch_sparse_mla(const CUtensorMap& qmap, const MlaParams& p, cudaStream_t st);

}  // namespace dsa

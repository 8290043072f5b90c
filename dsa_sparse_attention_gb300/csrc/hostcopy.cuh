// hostcopy.cuh — the copy kernel of the host-buffer layer step (hostcopy.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace dsa {

// Byte ranges copied by one host_copy launch (hostcopy.cu): device addresses on
// both sides (a page-locked host buffer through its mapped device pointer).
constexpr int kHostCopyMaxSegs = 8;
struct HostCopySeg {
  uint8_t* dst;
  const uint8_t* src;
  uint64_t bytes;
};
struct HostCopyParams {
  HostCopySeg seg[kHostCopyMaxSegs];
  int nseg;
};
cudaError_t launch_host_copy(const HostCopyParams& p, int num_sms, cudaStream_t st, bool chained);

}  // namespace dsa

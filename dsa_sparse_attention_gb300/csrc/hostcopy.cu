// hostcopy.cu — the transfers of the host-buffer layer step, done by SMs.
//
// On a GB300 the host's memory sits behind the chip-to-chip link and page-locked
// buffers are mapped into the GPU's address space.  Copy engines and SM loads
// both move about 200 GB/s over the link on large transfers; for the ~1 MB of a
// step's inputs or outputs the kernel saves the copy engine's start-up and, as a
// kernel, lets the scorer (chained by programmatic launch) set up while it runs
// (measured ~1.5 µs per direction against cudaMemcpyAsync in the same graph).
// The kernel below copies up to kHostCopyMaxSegs byte ranges in one launch, in
// either direction: the host side is addressed through its mapped device
// pointer, which the host code obtains (and range-checks) before it asks for a
// kernel copy.
#include <cuda_runtime.h>

#include "hostcopy.cuh"
#include "params.cuh"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;   // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kCopyThreads) host_copy_kernel(const __grid_constant__ HostCopyParams p) {
  // the next chained kernel may be scheduled now: its set-up overlaps the copy,
  // and its own dependency wait still waits for this grid to finish
  grid_dep_launch();
  grid_dep_wait();   // chained after a kernel that writes the source (or reads the destination)
  const uint64_t tid = uint64_t(blockIdx.x) * kCopyThreads + threadIdx.x;
  const uint64_t nth = uint64_t(gridDim.x) * kCopyThreads;
  for (int s = 0; s < p.nseg; ++s) {
    const HostCopySeg g = p.seg[s];
    const bool vec = ((reinterpret_cast<uintptr_t>(g.dst) | reinterpret_cast<uintptr_t>(g.src)) & 15) == 0;
    const uint64_t n16 = vec ? g.bytes / 16 : 0;
    const uint4* src = reinterpret_cast<const uint4*>(g.src);
    uint4* dst = reinterpret_cast<uint4*>(g.dst);
    for (uint64_t i = tid; i < n16; i += kCopyUnroll * nth) {
      uint4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (i + u * nth < n16) v[u] = src[i + u * nth];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (i + u * nth < n16) dst[i + u * nth] = v[u];
    }
    // the bytes past the last whole 16 (or all of them when either side is unaligned)
    for (uint64_t i = n16 * 16 + tid; i < g.bytes; i += nth) g.dst[i] = g.src[i];
  }
}

}  // namespace

cudaError_t launch_host_copy(const HostCopyParams& p, int num_sms, cudaStream_t st, bool chained) {
  uint64_t vecs = 0;
  for (int s = 0; s < p.nseg; ++s) vecs += (p.seg[s].bytes + 15) / 16;
  if (vecs == 0) return cudaSuccess;
  // one 16-byte transfer per thread where the bytes allow, at most one CTA per SM (the
  // chained scorer needs the rest of each SM's registers to be scheduled beside it)
  const uint64_t want = (vecs + kCopyThreads - 1) / kCopyThreads;
  const unsigned grid = static_cast<unsigned>(want < uint64_t(num_sms) ? want : uint64_t(num_sms));
  return launch_ex(host_copy_kernel, dim3(grid), dim3(kCopyThreads), 0, st, chained, 0u, p);
}

}  // namespace dsa

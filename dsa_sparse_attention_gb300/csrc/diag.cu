// diag.cu — dsa_selftest_wait_timeout: the bounded-wait path, made to run out.
//
// Every wait inside the warp-specialised kernels (scorer, attention) goes
// through mbar_wait / mbar_wait_inline, which give up after a limit, record
// DEV_TIMEOUT in the status word and set the CTA's abort flag so that the
// CTA's other waits return at once.  A healthy pipeline never reaches the
// limit, so this entry point runs the same helper on an mbarrier that nothing
// completes, with a short limit chosen by the caller: the wait must give up,
// the status word must carry the timeout, and the kernel must return on its
// own (the context stays usable).  Nothing is copied and no tensor-core work
// is in flight, so giving up leaves nothing behind.
#include "../../include/dsa.h"
#include "params.cuh"

namespace dsa {
dsa_status record_cuda_status(cudaError_t e);   // capi.cu
}

namespace {

using namespace dsa;

// One warp.  Lane 0 waits twice on a barrier nothing arrives on: the first wait
// runs into its limit, the second finds the abort flag set and returns without
// waiting.  A wait that reported success would be a logic error, recorded as a
// range finding so that the caller sees something other than the timeout.
__global__ void wait_timeout_kernel(uint32_t* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abortf;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abortf = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Abort ab{&abortf, status};
    const bool first = mbar_wait(&bar, 0, ab, limit);
    const long long t0 = clock64();
    const bool second = mbar_wait(&bar, 0, ab, limit);
    const bool second_fast = clock64() - t0 < limit;
    if (first || second || !second_fast || abortf == 0) atomicOr(status, DEV_BAD_BATCH);
  }
}

}  // namespace

extern "C" dsa_status dsa_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_cycles,
                                                dsa_stream_t stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || workspace_bytes < 256)
    return DSA_ERR_WORKSPACE;
  if (limit_cycles < 1000 || limit_cycles > kWaitLimitCycles) return DSA_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<uint32_t*>(workspace), static_cast<long long>(limit_cycles));
  return record_cuda_status(cudaGetLastError());
}

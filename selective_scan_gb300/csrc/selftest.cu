// Failure-detection self-test of the bounded mbarrier wait that every tensor-core
// kernel uses: one CTA waits on a barrier that nothing arrives at, with the same
// helpers and limit as the kernels. The wait must give up, raise the CTA's abort flag
// and let the kernel return, leaving the context usable. No trap, no fault, no
// endless loop: the outcome is a status word the host reads.
#include <cuda.h>

#include "common.cuh"

namespace mamba2 {
namespace {

#include "tc.cuh"

// status: 1 = the phase completed (impossible here), 2 = the wait gave up and raised
// the abort flag (the expected outcome), 3 = gave up without raising it
__global__ void bounded_wait_probe_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar_mem;
  __shared__ uint32_t abort_flag;
  const uint32_t bar = su32(&bar_mem);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool done = warp_wait(bar, 0u, &abort_flag);  // nothing arrives on phase 0
  if (threadIdx.x == 0) *status = done ? 1 : (abort_flag ? 2 : 3);
}

}  // namespace

cudaError_t launch_bounded_wait_probe(int32_t* status, cudaStream_t st) {
  bounded_wait_probe_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

}  // namespace mamba2

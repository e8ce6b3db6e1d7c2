// Self-check of the failure path shared by every pipeline wait (csa2_check_bounded_wait).
//
// The kernels' mbarrier waits are bounded by wall time: a wait that gives up sets
// CSA2_DEV_PIPELINE_TIMEOUT in the caller's status word, and the kernel drains and
// returns instead of spinning. This kernel makes that path run on purpose without
// touching a pipeline: one CTA waits, through the same helper, on an mbarrier that
// nothing arrives on, with the caller's (short) bound.
#include "csa2_internal.cuh"

namespace csa2 {

__global__ void __launch_bounds__(32) wait_check_kernel(uint64_t limit_ns, uint32_t* __restrict__ status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  // phase 0 of a fresh barrier completes only after one arrival, and none comes
  const bool ok = mbar_wait(a, 0, limit_ns);
  if (threadIdx.x == 0 && !ok) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
}

cudaError_t launch_wait_check(uint64_t limit_ns, uint32_t* status, cudaStream_t st) {
  wait_check_kernel<<<1, 32, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace csa2

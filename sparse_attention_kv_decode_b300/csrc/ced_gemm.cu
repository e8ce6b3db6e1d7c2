// CED KV projection (placeholder until the tcgen05 GEMM lands).
#include "csa2_internal.cuh"

namespace csa2 {
cudaError_t launch_ced_project(const void*, int64_t, int, const void*, const void*, int, uint8_t*,
                               uint8_t*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace csa2

// k_gemm_tc.cu -- tcgen05 GEMM (placeholder until the tensor-core kernel lands).
#include "common.cuh"
#include "internal.h"

namespace dfl {
bool gemm_tc_supported(const GemmDesc&) { return false; }
size_t gemm_tc_workspace(const GemmDesc&, int) { return 0; }
cudaError_t launch_gemm_tc(const GemmDesc&, void*, size_t, uint32_t*, uint32_t*, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace dfl

// gemm_bf16.cu -- bf16 instantiations of the tcgen05 GEMM (kind::f16, fp32 accumulation).
#include "gemm_kernel.cuh"
#include "gemm_pair.cuh"

namespace mmdit {
cudaError_t launch_gemm_bf16(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  return dispatch_gemm<kKindF16>(p, status, stream);
}
}  // namespace mmdit

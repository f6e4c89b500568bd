// gemm_tf32.cu -- fp32-operand instantiations of the tcgen05 GEMM (kind::tf32, fp32 accumulation).
#include "gemm_kernel.cuh"

namespace mmdit {
cudaError_t launch_gemm_tf32(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  return dispatch_gemm<kKindTF32>(p, status, stream);
}
}  // namespace mmdit

// gemm_fp8.cu -- E4M3 instantiations of the tcgen05 GEMM (kind::f8f6f4, fp32 accumulation).
// Operands are E4M3 codes of x * scale_x and W * scale_w ("FP8 training for Flux models",
// §Configuration, FP8 model configuration); the epilogue first divides the accumulator by
// scale_x * scale_w, then applies the bf16 epilogue of the linear it replaces.
#include "gemm_kernel.cuh"
#include "gemm_pair.cuh"

namespace mmdit {
cudaError_t launch_gemm_fp8(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  if (p.ep.bw_sx) return launch_gemm_blockwise(p, status, stream);  // blockwise recipe: per-tile scales
  if (p.N % 128 != 0 || p.K % 16 != 0 || p.a_mn || p.b_mn) return cudaErrorInvalidValue;
  if (!p.ep.scale_a || !p.ep.scale_w || (p.M1 > 0 && (!p.ep1.scale_a || !p.ep1.scale_w)))
    return cudaErrorInvalidValue;
  const bool wide = p.N % 256 == 0;
  if (p.act == 3) {
    // E5M2 A (the hybrid recipe's gradient) with E4M3 B: the backward's plain products only
    if (p.epi != kEpiBias) return cudaErrorInvalidValue;
    return wide ? run_gemm<kKindF8E5M2, 256, kEpiBias>(p, status, stream)
                : run_gemm<kKindF8E5M2, 128, kEpiBias>(p, status, stream);
  }
  if (use_pair(p)) {
    switch (p.epi) {
      case kEpiQkv: return run_gemm_pair<kKindF8, 256, kEpiQkv>(p, status, stream);
      case kEpiGateResid: return run_gemm_pair<kKindF8, 256, kEpiGateResid>(p, status, stream);
      case kEpiGeluF8: return run_gemm_pair<kKindF8, 256, kEpiGeluF8>(p, status, stream);
      case kEpiGelu: return run_gemm_pair<kKindF8, 256, kEpiGelu>(p, status, stream);  // tensorwise
      default: break;
    }
  }
  switch (p.epi) {
    case kEpiQkv:
      if (wide && p.ep.hidden % 256 == 0) return run_gemm<kKindF8, 256, kEpiQkv>(p, status, stream);
      return run_gemm<kKindF8, 128, kEpiQkv>(p, status, stream);
    case kEpiGateResid:
      return wide ? run_gemm<kKindF8, 256, kEpiGateResid>(p, status, stream)
                  : run_gemm<kKindF8, 128, kEpiGateResid>(p, status, stream);
    case kEpiGeluF8:
      return wide ? run_gemm<kKindF8, 256, kEpiGeluF8>(p, status, stream)
                  : run_gemm<kKindF8, 128, kEpiGeluF8>(p, status, stream);
    case kEpiGelu:  // tensorwise scaling: the bf16 GELU output is cast after its amax is taken
      return wide ? run_gemm<kKindF8, 256, kEpiGelu>(p, status, stream)
                  : run_gemm<kKindF8, 128, kEpiGelu>(p, status, stream);
    case kEpiBias:
      return wide ? run_gemm<kKindF8, 256, kEpiBias>(p, status, stream)
                  : run_gemm<kKindF8, 128, kEpiBias>(p, status, stream);
    default:
      return cudaErrorInvalidValue;
  }
}
}  // namespace mmdit

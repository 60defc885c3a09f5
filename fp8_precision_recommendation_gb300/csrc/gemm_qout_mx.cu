// Instantiations of the fused GEMM + normalization kernel whose epilogue
// also quantizes its bf16 output rows to E4M3 (per-row or MX 1x32 scales)
// for the next layer, for MX 1x32 E4M3 operands.
#include "gemm_norm.cuh"

namespace loka {

cudaError_t launch_gemm_qout_mx(GemmParams& p, int N, int sms, cudaStream_t stream) {
  return launch_kind<static_cast<int>(OperandKind::kMxE4M3), static_cast<int>(OutKind::kQuant)>(p, N, sms, stream);
}

}  // namespace loka

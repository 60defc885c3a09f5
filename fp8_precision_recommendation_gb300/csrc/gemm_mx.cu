// Instantiations of the fused GEMM + normalization kernel for MX 1x32 E4M3
// operands with E8M0 block scales, with bf16 or fp32 output.
#include "gemm_norm.cuh"

namespace loka {

cudaError_t launch_gemm_mx(GemmParams& p, int N, OutKind out, int sms, cudaStream_t stream) {
  constexpr int op = static_cast<int>(OperandKind::kMxE4M3);
  if (out == OutKind::kBf16) return launch_kind<op, static_cast<int>(OutKind::kBf16)>(p, N, sms, stream);
  if (out == OutKind::kF32) return launch_kind<op, static_cast<int>(OutKind::kF32)>(p, N, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace loka

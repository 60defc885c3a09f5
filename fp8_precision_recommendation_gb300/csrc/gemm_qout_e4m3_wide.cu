// Instantiations of the fused GEMM + normalization kernel whose epilogue
// also quantizes its bf16 output rows to E4M3 (per-row or MX 1x32 scales)
// for the next layer: E4M3 operands (per-tensor and per-row scales),
// rows of 512 to 2048 columns (thread-block clusters).
#include "gemm_norm.cuh"

namespace loka {

cudaError_t launch_gemm_qout_e4m3_wide(GemmParams& p, int N, int sms, cudaStream_t stream) {
  constexpr int op = static_cast<int>(OperandKind::kE4M3);
  return launch_wide<op, static_cast<int>(OutKind::kQuant)>(p, N, sms, stream);
}

}  // namespace loka

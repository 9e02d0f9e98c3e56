// Test build only: instantiations of the grouped GEMM kernel as a standalone GEMM1 with the
// plain epilogues of moe_test_gemm1 (FP32 pre-activations, BF16 intermediate) for the
// RELU2, GELU and RELU activations.
#include "gemm_plain.cuh"

namespace moe {
namespace gemm {

moe_status_t launch_plain_a(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem, cudaStream_t s) {
  switch (act) {
    case MOE_ACT_RELU2:
      if (mode == kG1Act) return launch_kernel<kG1Act, MOE_ACT_RELU2>(prm, units_max, smem, s);
      if (mode == kG1Preact) return launch_kernel<kG1Preact, MOE_ACT_RELU2>(prm, units_max, smem, s);
      break;
    case MOE_ACT_GELU:
      if (mode == kG1Act) return launch_kernel<kG1Act, MOE_ACT_GELU>(prm, units_max, smem, s);
      if (mode == kG1Preact) return launch_kernel<kG1Preact, MOE_ACT_RELU2>(prm, units_max, smem, s);
      break;
    case MOE_ACT_RELU:
      if (mode == kG1Act) return launch_kernel<kG1Act, MOE_ACT_RELU>(prm, units_max, smem, s);
      if (mode == kG1Preact) return launch_kernel<kG1Preact, MOE_ACT_RELU2>(prm, units_max, smem, s);
      break;
    default: break;
  }
  return MOE_ERR_INVALID_ARGUMENT;
}

}  // namespace gemm
}  // namespace moe

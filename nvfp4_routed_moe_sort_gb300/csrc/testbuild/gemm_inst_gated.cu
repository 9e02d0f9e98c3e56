// Test build only: instantiations of the grouped GEMM kernel as a standalone GEMM1 with the
// plain epilogues of moe_test_gemm1 (FP32 pre-activations, BF16 intermediate) for the
// SWIGLU and GEGLU activations.
#include "gemm_plain.cuh"

namespace moe {
namespace gemm {

moe_status_t launch_gated(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem, cudaStream_t s) {
  switch (act) {
    case MOE_ACT_SWIGLU:
      if (mode == kG1Act) return launch_kernel<kG1Act, MOE_ACT_SWIGLU>(prm, units_max, smem, s);
      if (mode == kG1Preact) return launch_kernel<kG1Preact, MOE_ACT_SWIGLU>(prm, units_max, smem, s);
      break;
    case MOE_ACT_GEGLU:
      if (mode == kG1Act) return launch_kernel<kG1Act, MOE_ACT_GEGLU>(prm, units_max, smem, s);
      if (mode == kG1Preact) return launch_kernel<kG1Preact, MOE_ACT_SWIGLU>(prm, units_max, smem, s);
      break;
    default: break;
  }
  return MOE_ERR_INVALID_ARGUMENT;
}

}  // namespace gemm
}  // namespace moe

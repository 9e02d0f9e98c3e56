// Instantiations of the grouped GEMM kernel: GEMM2 with BF16 expert rows, and GEMM2 adding
// route-weighted rows into an FP32 accumulator.
#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

moe_status_t launch_rows(int mode, const GemmParams& prm, int64_t units_max, size_t smem, cudaStream_t s) {
  if (mode == kG2Reduce) return launch_kernel<kG2Reduce, MOE_ACT_IDENTITY>(prm, units_max, smem, s);
  return launch_kernel<kG2Rows, MOE_ACT_IDENTITY>(prm, units_max, smem, s);
}

}  // namespace gemm
}  // namespace moe

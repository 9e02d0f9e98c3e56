// Instantiation of the grouped GEMM kernel: GEMM2 with BF16 expert rows.
#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

moe_status_t launch_rows(const GemmParams& prm, int64_t units_max, size_t smem, cudaStream_t s) {
  return launch_kernel<kG2Rows, MOE_ACT_IDENTITY>(prm, units_max, smem, s);
}

}  // namespace gemm
}  // namespace moe

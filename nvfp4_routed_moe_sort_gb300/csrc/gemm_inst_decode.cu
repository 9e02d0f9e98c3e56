// Instantiations of the decode-shaped chained GEMM kernel for every activation.
#include "gemm_decode.cuh"

namespace moe {
namespace dgemm {

moe_status_t launch_act(bool rows, int act, const Params& prm, int grid, size_t smem, cudaStream_t s) {
  switch (act) {
    case MOE_ACT_SWIGLU:
      return rows ? launch_kernel<true, MOE_ACT_SWIGLU>(prm, grid, smem, s) : launch_kernel<false, MOE_ACT_SWIGLU>(prm, grid, smem, s);
    case MOE_ACT_RELU2:
      return rows ? launch_kernel<true, MOE_ACT_RELU2>(prm, grid, smem, s) : launch_kernel<false, MOE_ACT_RELU2>(prm, grid, smem, s);
    case MOE_ACT_GEGLU:
      return rows ? launch_kernel<true, MOE_ACT_GEGLU>(prm, grid, smem, s) : launch_kernel<false, MOE_ACT_GEGLU>(prm, grid, smem, s);
    case MOE_ACT_GELU:
      return rows ? launch_kernel<true, MOE_ACT_GELU>(prm, grid, smem, s) : launch_kernel<false, MOE_ACT_GELU>(prm, grid, smem, s);
    case MOE_ACT_RELU:
      return rows ? launch_kernel<true, MOE_ACT_RELU>(prm, grid, smem, s) : launch_kernel<false, MOE_ACT_RELU>(prm, grid, smem, s);
    case MOE_ACT_SILU:
      return rows ? launch_kernel<true, MOE_ACT_SILU>(prm, grid, smem, s) : launch_kernel<false, MOE_ACT_SILU>(prm, grid, smem, s);
    case MOE_ACT_IDENTITY:
      return rows ? launch_kernel<true, MOE_ACT_IDENTITY>(prm, grid, smem, s) : launch_kernel<false, MOE_ACT_IDENTITY>(prm, grid, smem, s);
    default: return MOE_ERR_INVALID_ARGUMENT;
  }
}

}  // namespace dgemm
}  // namespace moe

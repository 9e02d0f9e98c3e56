// Instantiations of the grouped GEMM kernel: GEMM1 and GEMM2 chained in one launch, with the
// SILU, IDENTITY activations.
#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

moe_status_t launch_chain_plain_b(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem,
                              cudaStream_t s) {
  switch (act) {
    case MOE_ACT_SILU:
      return mode == kChainReduce ? launch_kernel<kChainReduce, MOE_ACT_SILU>(prm, units_max, smem, s)
                                  : launch_kernel<kChainRows, MOE_ACT_SILU>(prm, units_max, smem, s);
    case MOE_ACT_IDENTITY:
      return mode == kChainReduce ? launch_kernel<kChainReduce, MOE_ACT_IDENTITY>(prm, units_max, smem, s)
                                  : launch_kernel<kChainRows, MOE_ACT_IDENTITY>(prm, units_max, smem, s);
    default: return MOE_ERR_INVALID_ARGUMENT;
  }
}

}  // namespace gemm
}  // namespace moe

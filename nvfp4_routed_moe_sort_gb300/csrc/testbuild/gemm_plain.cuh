// Test build only: the standalone GEMM1 launchers with plain epilogues (FP32 pre-activations,
// BF16 intermediate), instantiated in this folder's gemm_inst_*.cu files.
#pragma once

#include "../gemm_kernel.cuh"

namespace moe {
namespace gemm {

moe_status_t launch_gated(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem, cudaStream_t s);
moe_status_t launch_plain_a(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem,
                            cudaStream_t s);
moe_status_t launch_plain_b(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem,
                            cudaStream_t s);

}  // namespace gemm
}  // namespace moe

// Test build only (libmoe_nvfp4_test.so): the entry points of include/moe_nvfp4_test.h.
//
// They reach paths that normal inputs never take: a standalone GEMM1 with plain epilogues
// (FP32 pre-activations, BF16 intermediate), the decode GEMM's scheduling fallbacks, and the
// GEMM kernels' bounded waits running out. Every option is an argument; nothing here keeps
// state between calls.
#include <string.h>

#include "../../../include/moe_nvfp4_test.h"
#include "gemm_plain.cuh"

namespace moe {
namespace {

using namespace gemm;

TestOptions to_internal(const moe_test_options_t* o) {
  TestOptions t;
  if (o != nullptr) {
    t.decode_hooks = o->decode_hooks;
    t.wait_limit_ns = o->wait_limit_ns;
    t.withhold_release = o->withhold_release;
  }
  return t;
}

// one GEMM1 on its own with a plain epilogue (kG1Preact or kG1Act)
moe_status_t launch_gemm1_plain(const GemmLaunch& g, cudaStream_t s) {
  if (g.cap == 0) return MOE_OK;
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  if (!fill_phase(prm.ph[0], g)) return MOE_ERR_CUDA;
  fill_common(prm, g);
  prm.sparse = 0;
  prm.wait_ns = kWaitLimitNs;
  const int64_t units_max = (g.cap / kTileM) * prm.ph[0].n_tiles;
  const size_t smem = smem_bytes(g.El, false);
  switch (g.act) {
    case MOE_ACT_SWIGLU:
    case MOE_ACT_GEGLU: return launch_gated(g.mode, g.act, prm, units_max, smem, s);
    case MOE_ACT_RELU2:
    case MOE_ACT_GELU:
    case MOE_ACT_RELU: return launch_plain_a(g.mode, g.act, prm, units_max, smem, s);
    case MOE_ACT_SILU:
    case MOE_ACT_IDENTITY: return launch_plain_b(g.mode, g.act, prm, units_max, smem, s);
    default: return MOE_ERR_INVALID_ARGUMENT;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_test_options_t moe_test_default_options(void) {
  const TestOptions t;
  moe_test_options_t o;
  o.decode_hooks = t.decode_hooks;
  o.withhold_release = t.withhold_release;
  o.wait_limit_ns = t.wait_limit_ns;
  return o;
}

extern "C" moe_status_t moe_test_routed_forward(const uint16_t* x, int32_t M, int64_t ld_x, int32_t act_scale_mode,
                                                const int32_t* topk_ids, int32_t topk_ids_format, int32_t top_k,
                                                int32_t num_experts, int32_t local_expert_offset,
                                                const void* topk_weights, int32_t topk_weights_dtype,
                                                float routed_scaling_factor, const moe_nvfp4_weights_t* w,
                                                const void* prepared, size_t prepared_bytes, float fc2_input_scale,
                                                int32_t do_finalize, uint16_t* out, uint16_t* gemm2_out,
                                                int32_t* token_to_row, void* workspace, size_t workspace_bytes,
                                                int32_t* dev_status, void* const* step_events,
                                                int32_t num_step_events, const moe_test_options_t* options,
                                                moe_stream_t stream) {
  MOE_CHECK(options == nullptr || options->wait_limit_ns > 0, MOE_ERR_INVALID_ARGUMENT);
  return routed_forward(x, M, ld_x, act_scale_mode, topk_ids, topk_ids_format, top_k, num_experts,
                        local_expert_offset, topk_weights, topk_weights_dtype, routed_scaling_factor, w, prepared,
                        prepared_bytes, fc2_input_scale, do_finalize, out, gemm2_out, token_to_row, workspace,
                        workspace_bytes, dev_status, step_events, num_step_events, to_internal(options), stream);
}

extern "C" moe_status_t moe_test_gemm1(const int32_t* padded_offsets, const int32_t* row_to_slot, int32_t M,
                                       int32_t top_k, const uint8_t* xq, const uint8_t* xsf, const float* xs,
                                       const moe_nvfp4_weights_t* w, const void* prepared, size_t prepared_bytes,
                                       int32_t mode, void* dbg_out, void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, moe_stream_t stream) {
  moe_status_t st = check_weights(w);
  if (st != MOE_OK) return st;
  MOE_CHECK(M >= 0 && top_k >= 1 && (mode == 0 || mode == 1), MOE_ERR_INVALID_ARGUMENT);
  const Dims d = make_dims(w);
  const WorkspaceLayout L = workspace_layout(d, M, top_k, MOE_OUTPUT_UNFINALIZED);
  st = check_forward_common(padded_offsets, row_to_slot, M, top_k, xq, xsf, xs, w, prepared, prepared_bytes,
                            workspace, workspace_bytes, dev_status, L.total);
  if (st != MOE_OK) return st;
  if (M == 0) return MOE_OK;
  MOE_CHECK(dbg_out != nullptr, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(dbg_out), MOE_ERR_MISALIGNED);
  cudaStream_t s = as_stream(stream);
  const Bufs b = carve(workspace, L);
  const Prepared pw = prepared_ptrs(prepared, prepared_layout(d));
  st = launch_permute(padded_offsets, static_cast<int>(d.El), row_to_slot, top_k, L.cap, xq, xsf,
                      static_cast<int>(d.H), b.aq, b.asf, b.sched, b.mtd, counter_ints(L, L.mtd), nullptr, nullptr, 0,
                      s);
  if (st != MOE_OK) return st;
  GemmLaunch g1 = gemm1_launch(d, L, b, pw, padded_offsets, row_to_slot, xs, top_k, dev_status);
  g1.mode = mode == 0 ? kG1Preact : kG1Act;
  g1.out = dbg_out;
  g1.out_sf = nullptr;
  return launch_gemm1_plain(g1, s);
}

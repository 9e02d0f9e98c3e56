// C ABI: argument validation, buffer carving and the launch sequence of the forward.
//
// Sources: FlashInfer flashinfer.fused_moe.CudnnGroupedGemmNvfp4Config (pipeline order:
// permutation, GEMM1, activation, GEMM2, finalize; MoEFinalizeConfig(do_finalize=False));
// FlashInfer flashinfer.fused_moe.alphamoe_nvfp4_aligned_moe (16-byte alignment of
// pointers and row strides; out must not overlap an input); Megatron-Core
// core.inference.moe.flashinfer_nvfp4 (prepare_routed_nvfp4_weights, in-place refresh).
#include <math.h>

#include "common.cuh"
#include "host_util.h"
#include "layout.h"

using namespace moe;

namespace {

bool valid_output_mode(int32_t m) { return m >= MOE_OUTPUT_UNFINALIZED && m <= MOE_OUTPUT_ACCUMULATE; }

}  // namespace

moe_status_t moe::check_weights(const moe_nvfp4_weights_t* w) {
  MOE_CHECK(w != nullptr, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(w->activation >= MOE_ACT_SWIGLU && w->activation <= MOE_ACT_IDENTITY, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(w->num_local_experts >= 1 && w->hidden > 0 && w->inter > 0, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(w->num_local_experts <= kMaxLocalExperts, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(w->hidden % 128 == 0 && w->inter % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(w->hidden <= 65536 && w->inter <= 65536, MOE_ERR_UNSUPPORTED_SHAPE);
  return MOE_OK;
}

namespace moe {

Bufs carve(void* ws, const WorkspaceLayout& L) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  Bufs r;
  r.sched = reinterpret_cast<int32_t*>(b + L.sched);
  r.mtd = reinterpret_cast<int32_t*>(b + L.mtd);
  r.aq = b + L.aq;
  r.asf = b + L.asf;
  r.iq = b + L.iq;
  r.isf = b + L.isf;
  r.g = L.g ? reinterpret_cast<uint16_t*>(b + L.g) : nullptr;
  return r;
}

Prepared prepared_ptrs(const void* prepared, const PreparedLayout& L) {
  const uint8_t* b = static_cast<const uint8_t*>(prepared);
  return {b + L.w1, b + L.w1sf, b + L.w2, b + L.w2sf, reinterpret_cast<const float*>(b + L.a1),
          reinterpret_cast<const float*>(b + L.a2), reinterpret_cast<const float*>(b + L.a1g)};
}

// checks shared by the forward and the GEMM1 test hook
moe_status_t check_forward_common(const int32_t* padded_offsets, const int32_t* row_to_slot, int32_t M,
                                  int32_t top_k, const uint8_t* xq, const uint8_t* xsf, const float* xs,
                                  const moe_nvfp4_weights_t* w, const void* prepared, size_t prepared_bytes,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status, size_t ws_need) {
  moe_status_t st = check_weights(w);
  if (st != MOE_OK) return st;
  MOE_CHECK(M >= 0 && top_k >= 1 && top_k <= w->num_local_experts * 64, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(static_cast<int64_t>(M) * top_k < (int64_t(1) << 30), MOE_ERR_UNSUPPORTED_SHAPE);
  const Dims d = make_dims(w);
  MOE_CHECK(prepared != nullptr && prepared_bytes >= prepared_layout(d).total, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(prepared), MOE_ERR_MISALIGNED);
  MOE_CHECK(workspace_bytes >= ws_need, MOE_ERR_WORKSPACE_TOO_SMALL);
  if (M == 0) return MOE_OK;
  MOE_CHECK(padded_offsets && row_to_slot && xq && xsf && xs && dev_status && workspace, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(padded_offsets) && aligned16(row_to_slot) && aligned16(xq) && aligned16(xsf) &&
                aligned16(xs) && aligned16(dev_status) && aligned16(workspace),
            MOE_ERR_MISALIGNED);
  return MOE_OK;
}

GemmLaunch gemm1_launch(const Dims& d, const WorkspaceLayout& L, const Bufs& b, const Prepared& pw,
                        const int32_t* padded_offsets, const int32_t* row_to_slot, const float* xs, int top_k,
                        int32_t* dev_status) {
  GemmLaunch g;
  g.a = b.aq;
  g.a_sf = b.asf;
  g.b = pw.w1;
  g.b_sf = pw.w1sf;
  g.alpha = pw.a1;
  g.alpha_gate = pw.a1g;
  g.xs = xs;
  g.padded_offsets = padded_offsets;
  g.row_to_slot = row_to_slot;
  g.cap = L.cap;
  g.El = d.El;
  g.K = d.H;
  g.Kp = d.Hp;
  g.N = d.N1;
  g.Np = d.N1p;
  g.top_k = top_k;
  g.inter = static_cast<int>(d.I);
  g.gated = d.gated;
  g.act = d.act;
  g.g2 = 1.0f;
  g.out = b.iq;
  g.out_sf = b.isf;
  g.dev_status = dev_status;
  g.tile_counter = b.sched;
  g.mode = kG1Fused;
  return g;
}

}  // namespace moe

extern "C" const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARGUMENT: return "MOE_ERR_INVALID_ARGUMENT";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_OVERLAP: return "MOE_ERR_OVERLAP";
    default: return "MOE_ERR_UNKNOWN";
  }
}

extern "C" int32_t moe_abi_version(void) { return MOE_NVFP4_ABI_VERSION; }

extern "C" size_t moe_prepared_weights_bytes(const moe_nvfp4_weights_t* w) {
  if (check_weights(w) != MOE_OK) return 0;
  return prepared_layout(make_dims(w)).total;
}

extern "C" moe_status_t moe_prepare_weights(const moe_nvfp4_weights_t* w, void* prepared, size_t prepared_bytes,
                                            moe_stream_t stream) {
  moe_status_t st = check_weights(w);
  if (st != MOE_OK) return st;
  MOE_CHECK(w->w1 && w->w1_sf && w->w1_alpha && w->w2 && w->w2_sf && w->w2_alpha && prepared,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(w->w1) && aligned16(w->w1_sf) && aligned16(w->w1_alpha) && aligned16(w->w2) &&
                aligned16(w->w2_sf) && aligned16(w->w2_alpha) && aligned16(prepared) &&
                (w->w1_gate_alpha == nullptr || aligned16(w->w1_gate_alpha)),
            MOE_ERR_MISALIGNED);
  const Dims d = make_dims(w);
  const PreparedLayout L = prepared_layout(d);
  MOE_CHECK(prepared_bytes >= L.total, MOE_ERR_WORKSPACE_TOO_SMALL);
  MOE_CHECK(!overlaps(prepared, L.total, w->w1, d.El * d.N1 * d.H / 2) &&
                !overlaps(prepared, L.total, w->w2, d.El * d.H * d.I / 2),
            MOE_ERR_OVERLAP);
  cudaStream_t s = as_stream(stream);
  uint8_t* b = static_cast<uint8_t*>(prepared);
  st = launch_prepare_matrix(w->w1, w->w1_sf, static_cast<int>(d.El), static_cast<int>(d.N1),
                             static_cast<int>(d.N1p), static_cast<int>(d.H), d.gated ? static_cast<int>(d.I) : 0,
                             b + L.w1, b + L.w1sf, s);
  if (st != MOE_OK) return st;
  st = launch_prepare_matrix(w->w2, w->w2_sf, static_cast<int>(d.El), static_cast<int>(d.H),
                             static_cast<int>(d.Hp), static_cast<int>(d.I), 0, b + L.w2, b + L.w2sf, s);
  if (st != MOE_OK) return st;
  MOE_CUDA(cudaMemcpyAsync(b + L.a1, w->w1_alpha, d.El * 4, cudaMemcpyDeviceToDevice, s));
  MOE_CUDA(cudaMemcpyAsync(b + L.a2, w->w2_alpha, d.El * 4, cudaMemcpyDeviceToDevice, s));
  MOE_CUDA(cudaMemcpyAsync(b + L.a1g, w->w1_gate_alpha ? w->w1_gate_alpha : w->w1_alpha, d.El * 4,
                           cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

extern "C" size_t moe_forward_workspace_bytes(int32_t M, int32_t top_k, const moe_nvfp4_weights_t* w,
                                              int32_t do_finalize) {
  if (check_weights(w) != MOE_OK || M < 0 || top_k < 1 || !valid_output_mode(do_finalize)) return 0;
  return workspace_layout(make_dims(w), M, top_k, do_finalize).total;
}

extern "C" moe_status_t moe_forward_workspace_layout(int32_t M, int32_t top_k, const moe_nvfp4_weights_t* w,
                                                     int32_t do_finalize, size_t offsets[6]) {
  moe_status_t st = check_weights(w);
  if (st != MOE_OK) return st;
  MOE_CHECK(M >= 0 && top_k >= 1 && offsets && valid_output_mode(do_finalize), MOE_ERR_INVALID_ARGUMENT);
  const WorkspaceLayout L = workspace_layout(make_dims(w), M, top_k, do_finalize);
  offsets[0] = L.aq;
  offsets[1] = L.asf;
  offsets[2] = L.iq;
  offsets[3] = L.isf;
  offsets[4] = L.g;
  offsets[5] = L.total;
  return MOE_OK;
}

namespace moe {

// The launches of one forward after validation: permute (unless a fused prologue already
// laid the rows out), GEMM1 with the fused activation and requant, GEMM2, and the combine.
moe_status_t forward_chain(const int32_t* padded_offsets, const int32_t* row_to_slot, const int32_t* token_to_row,
                           int32_t M, int32_t top_k, const uint8_t* xq, const uint8_t* xsf, const float* xs,
                           const moe_nvfp4_weights_t* w, const void* prepared, const void* topk_weights,
                           int32_t topk_weights_dtype, float routed_scaling_factor, float fc2_input_scale,
                           int32_t do_finalize, uint16_t* out, uint16_t* gemm2_out, void* workspace,
                           int32_t* dev_status, void* const* step_events, int32_t num_step_events, bool run_permute,
                           const RoutingHint& hint, const TestOptions& topt, cudaStream_t s) {
  const Dims d = make_dims(w);
  const bool fin = do_finalize == MOE_OUTPUT_FINALIZED;
  const bool accum = do_finalize == MOE_OUTPUT_ACCUMULATE;
  const WorkspaceLayout L = workspace_layout(d, M, top_k, do_finalize);
  const Bufs b = carve(workspace, L);
  uint16_t* rows_out = fin ? b.g : gemm2_out;
  float* acc = accum ? reinterpret_cast<float*>(b.g) : nullptr;
  const Prepared pw = prepared_ptrs(prepared, prepared_layout(d));
  // while the stream is being captured, the marks become external event-record nodes so the
  // caller can read their timestamps after each graph launch
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (num_step_events == 5) MOE_CUDA(cudaStreamIsCapturing(s, &capturing));
  auto mark = [&](int i) -> moe_status_t {
    if (num_step_events != 5) return MOE_OK;
    cudaEvent_t ev = static_cast<cudaEvent_t>(step_events[i]);
    if (capturing == cudaStreamCaptureStatusActive)
      MOE_CUDA(cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal));
    else
      MOE_CUDA(cudaEventRecord(ev, s));
    return MOE_OK;
  };
  moe_status_t st = MOE_OK;
  if ((st = mark(0)) != MOE_OK) return st;
  if (run_permute)
    st = launch_permute(padded_offsets, static_cast<int>(d.El), row_to_slot, top_k, L.cap, xq, xsf,
                        static_cast<int>(d.H), b.aq, b.asf, b.sched, b.mtd, counter_ints(L, L.mtd), accum ? out : nullptr,
                        acc, accum ? static_cast<int64_t>(M) * d.H : 0, s);
  if (st != MOE_OK) return st;
  if ((st = mark(1)) != MOE_OK) return st;
  GemmLaunch g1 = gemm1_launch(d, L, b, pw, padded_offsets, row_to_slot, xs, top_k, dev_status);
  g1.g2 = fc2_input_scale;
  // GEMM1 and GEMM2 in one chained launch (the GEMM2 mark then follows it)
  GemmLaunch g2;
  g2.mode = accum ? kG2Reduce : kG2Rows;
  g2.a = b.iq;
  g2.a_sf = b.isf;
  g2.b = pw.w2;
  g2.b_sf = pw.w2sf;
  g2.alpha = pw.a2;
  g2.alpha_gate = nullptr;
  g2.xs = nullptr;
  g2.padded_offsets = padded_offsets;
  g2.row_to_slot = row_to_slot;
  g2.cap = L.cap;
  g2.El = d.El;
  g2.K = d.I;
  g2.Kp = d.Ip;
  g2.N = d.H;
  g2.Np = d.Hp;
  g2.top_k = top_k;
  g2.inter = static_cast<int>(d.I);
  g2.gated = false;  // GEMM2 columns are plain output columns
  g2.act = MOE_ACT_IDENTITY;
  g2.g2 = fc2_input_scale;
  g2.out = accum ? static_cast<void*>(acc) : static_cast<void*>(rows_out);
  g2.out_sf = nullptr;
  g2.route_w = topk_weights;
  g2.route_w_dtype = topk_weights_dtype;
  g2.rsf = routed_scaling_factor;
  g2.dev_status = dev_status;
  g2.tile_counter = b.sched + 1;
  if (M <= kDecodeMaxTokens)
    st = launch_gemm_decode(g1, g2, reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + L.edone),
                            reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + L.own), hint, topt, s);
  else
    st = launch_gemm_chain(g1, g2, b.mtd, topt, s);
  if (st != MOE_OK) return st;
  if ((st = mark(2)) != MOE_OK) return st;
  if ((st = mark(3)) != MOE_OK) return st;
  if (fin) {
    st = launch_finalize(rows_out, topk_weights, topk_weights_dtype, routed_scaling_factor, token_to_row, M, top_k,
                         static_cast<int>(d.H), out, s);
    if (st != MOE_OK) return st;
  } else if (accum) {
    st = launch_store_acc(acc, static_cast<int64_t>(M) * d.H, out, s);
    if (st != MOE_OK) return st;
  }
  return mark(4);
}

}  // namespace moe

extern "C" moe_status_t moe_grouped_fp4_forward(const int32_t* padded_offsets, const int32_t* row_to_slot,
                                                const int32_t* token_to_row, int32_t M, int32_t top_k,
                                                const uint8_t* xq, const uint8_t* xsf, const float* xs,
                                                const moe_nvfp4_weights_t* w, const void* prepared,
                                                size_t prepared_bytes, const void* topk_weights,
                                                int32_t topk_weights_dtype, float routed_scaling_factor,
                                                float fc2_input_scale, int32_t do_finalize, uint16_t* out,
                                                uint16_t* gemm2_out, void* workspace, size_t workspace_bytes,
                                                int32_t* dev_status, void* const* step_events,
                                                int32_t num_step_events, moe_stream_t stream) {
  moe_status_t st = check_weights(w);
  if (st != MOE_OK) return st;
  MOE_CHECK(M >= 0 && top_k >= 1 && valid_output_mode(do_finalize), MOE_ERR_INVALID_ARGUMENT);
  const Dims d = make_dims(w);
  const bool fin = do_finalize == MOE_OUTPUT_FINALIZED;
  const bool accum = do_finalize == MOE_OUTPUT_ACCUMULATE;
  const WorkspaceLayout L = workspace_layout(d, M, top_k, do_finalize);
  st = check_forward_common(padded_offsets, row_to_slot, M, top_k, xq, xsf, xs, w, prepared, prepared_bytes,
                            workspace, workspace_bytes, dev_status, L.total);
  if (st != MOE_OK) return st;
  MOE_CHECK(isfinite(fc2_input_scale) && fc2_input_scale > 0.0f, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(isfinite(routed_scaling_factor), MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(topk_weights_dtype >= MOE_WEIGHTS_F32 && topk_weights_dtype <= MOE_WEIGHTS_PACKED,
            MOE_ERR_INVALID_ARGUMENT);
  const size_t wbytes = static_cast<size_t>(M) * top_k * (topk_weights_dtype == MOE_WEIGHTS_BF16 ? 2 : 4);
  MOE_CHECK(num_step_events == 0 || (num_step_events == 5 && step_events != nullptr), MOE_ERR_INVALID_ARGUMENT);
  if (M == 0) return MOE_OK;
  MOE_CHECK(token_to_row && topk_weights, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(token_to_row) && aligned16(topk_weights), MOE_ERR_MISALIGNED);
  if (fin || accum) {
    MOE_CHECK(out != nullptr, MOE_ERR_INVALID_ARGUMENT);
    MOE_CHECK(aligned16(out), MOE_ERR_MISALIGNED);
    const size_t ob = static_cast<size_t>(M) * d.H * 2;
    MOE_CHECK(!overlaps(out, ob, xq, static_cast<size_t>(M) * d.H / 2) &&
                  !overlaps(out, ob, xsf, static_cast<size_t>(M) * d.H / 16) &&
                  !overlaps(out, ob, xs, static_cast<size_t>(M) * 4) &&
                  !overlaps(out, ob, topk_weights, wbytes) &&
                  !overlaps(out, ob, token_to_row, static_cast<size_t>(M) * top_k * 4) &&
                  !overlaps(out, ob, workspace, L.total) && !overlaps(out, ob, prepared, prepared_bytes),
              MOE_ERR_OVERLAP);
  } else {
    MOE_CHECK(gemm2_out != nullptr, MOE_ERR_INVALID_ARGUMENT);
    MOE_CHECK(aligned16(gemm2_out), MOE_ERR_MISALIGNED);
    const size_t gb = static_cast<size_t>(L.cap) * d.H * 2;
    MOE_CHECK(!overlaps(gemm2_out, gb, workspace, L.total) && !overlaps(gemm2_out, gb, prepared, prepared_bytes) &&
                  !overlaps(gemm2_out, gb, xq, static_cast<size_t>(M) * d.H / 2),
              MOE_ERR_OVERLAP);
  }
  return forward_chain(padded_offsets, row_to_slot, token_to_row, M, top_k, xq, xsf, xs, w, prepared, topk_weights,
                       topk_weights_dtype, routed_scaling_factor, fc2_input_scale, do_finalize, out, gemm2_out,
                       workspace, dev_status, step_events, num_step_events, true, RoutingHint(), TestOptions(),
                       as_stream(stream));
}

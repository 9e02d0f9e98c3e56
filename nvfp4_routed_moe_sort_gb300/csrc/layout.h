// Host-side sizes and buffer layouts shared by the entry points, and the internal launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_nvfp4.h"
#include "common.cuh"

namespace moe {

// Problem sizes, with the paddings the kernels need: every GEMM tile reads 256 K values per
// stage and covers 256 output columns, so K dimensions and per-expert weight rows are padded
// to 256 (zero data, zero scales).
struct Dims {
  int64_t El, H, I, N1;
  bool gated;
  int act;
  int64_t N1p;  // W1 rows per expert in the prepared layout
  int64_t Hp;   // H padded to 256: GEMM1 K, and W2 rows per expert
  int64_t Ip;   // I padded to 256: GEMM2 K
};

inline Dims make_dims(const moe_nvfp4_weights_t* w) {
  Dims d;
  d.El = w->num_local_experts;
  d.H = w->hidden;
  d.I = w->inter;
  d.act = w->activation;
  d.gated = w->activation == MOE_ACT_SWIGLU || w->activation == MOE_ACT_GEGLU;
  d.N1 = d.gated ? 2 * d.I : d.I;
  d.N1p = roundup64(d.N1, kTileN);
  d.Hp = roundup64(d.H, kTileK);
  d.Ip = roundup64(d.I, kTileK);
  return d;
}

inline size_t take(size_t& cursor, size_t bytes) {
  const size_t at = cursor;
  cursor = static_cast<size_t>(roundup64(static_cast<int64_t>(cursor + bytes), 256));
  return at;
}

// Prepared weights: W1 data [El, N1p, H/2], W1 scale tiles [El][N1p/128][Hp/64][512],
// W2 data [El, Hp, I/2], W2 scale tiles [El][Hp/128][Ip/64][512], alpha1 [El], alpha2 [El],
// gate alpha1 [El] (the W1 gate rows' scalars; a copy of alpha1 unless given separately).
struct PreparedLayout {
  size_t w1, w1sf, w2, w2sf, a1, a2, a1g, total;
};

inline PreparedLayout prepared_layout(const Dims& d) {
  PreparedLayout L;
  size_t c = 0;
  L.w1 = take(c, d.El * d.N1p * d.H / 2);
  L.w1sf = take(c, d.El * d.N1p * d.Hp / 16);
  L.w2 = take(c, d.El * d.Hp * d.I / 2);
  L.w2sf = take(c, d.El * d.Hp * d.Ip / 16);
  L.a1 = take(c, d.El * 4);
  L.a2 = take(c, d.El * 4);
  L.a1g = take(c, d.El * 4);
  L.total = c;
  return L;
}

// Forward workspace: GEMM tile counters (256 B), permuted activations [cap, H/2] + scale tiles [cap/128][Hp/64][512],
// intermediate [cap, I/2] + scale tiles [cap/128][Ip/64][512], and the BF16 expert rows
// [cap, H] (finalized output) or the FP32 accumulator [M, H] (accumulated output).
// Ownership flags of the decode GEMM's statically assigned first units (one per CTA).
constexpr int64_t kOwnFlags = 1024;

struct WorkspaceLayout {
  size_t sched, mtd, edone, own, aq, asf, iq, isf, g, total;
  int64_t cap;
};

inline int64_t plan_capacity_rows(int64_t M, int64_t top_k, int64_t El) {
  const int64_t slots = M * top_k;
  const int64_t segs = slots < El ? slots : El;
  return roundup64(slots + (kSegAlign - 1) * segs, kSegAlign);
}

inline WorkspaceLayout workspace_layout(const Dims& d, int64_t M, int64_t top_k, int out_mode) {
  WorkspaceLayout L;
  L.cap = plan_capacity_rows(M, top_k, d.El);
  size_t c = 0;
  L.sched = take(c, 256);  // GEMM tile counters, zeroed by the permute kernel
  L.mtd = take(c, (L.cap / kTileM) * 4);  // per-row-tile GEMM1 completion counts (chained GEMMs), zeroed too
  L.edone = take(c, d.El * 4);            // per-expert GEMM1 completion counts (decode GEMMs), zeroed too
  L.own = take(c, kOwnFlags * 4);         // first-unit ownership flags (decode GEMMs), zeroed too
  L.aq = take(c, L.cap * d.H / 2);
  L.asf = take(c, L.cap * d.Hp / 16);
  L.iq = take(c, L.cap * d.I / 2);
  L.isf = take(c, L.cap * d.Ip / 16);
  L.g = out_mode == MOE_OUTPUT_FINALIZED     ? take(c, L.cap * d.H * 2)
        : out_mode == MOE_OUTPUT_ACCUMULATE ? take(c, M * d.H * 4)
                                            : 0;
  L.total = c;
  return L;
}

// ints from `from` (L.sched or L.mtd) through the last ownership flag: the counters that a
// forward zeroes before its GEMMs
inline int64_t counter_ints(const WorkspaceLayout& L, size_t from) {
  return static_cast<int64_t>(L.own - from) / 4 + kOwnFlags;
}

// The routing ids of the step, when the GEMMs are launched from the one-call path: the
// decode GEMM reads them before its dependency wait to start the first unit's weights.
struct RoutingHint {
  const int32_t* ids = nullptr;
  int32_t id_mask = -1;
  int32_t off = 0;
  int32_t slots = 0;
};

// GEMM epilogue modes
enum GemmMode : int {
  kG1Fused = 0,   // activation + NVFP4 requant of the intermediate
  kG1Preact = 1,  // FP32 pre-activations (test hook)
  kG1Act = 2,     // BF16 intermediate (test hook)
  kG2Rows = 3,    // BF16 expert rows
  kG2Reduce = 4,  // route-weighted rows added in FP32 into the [M, H] accumulator
  kChainRows = 5,    // GEMM1 (kG1Fused) then GEMM2 (kG2Rows) in one launch
  kChainReduce = 6,  // GEMM1 (kG1Fused) then GEMM2 (kG2Reduce) in one launch
};

// GEMM1 and GEMM2 run as one chained launch: the GEMM2 tiles of a row tile start once its
// GEMM1 tiles are written, so the second weight stream overlaps the first GEMM's tail
// instead of waiting for a kernel boundary. Batches of at most this many tokens (so at most
// 16 rows per expert) run the decode-shaped GEMMs: the weight tile is the MMA's M operand,
// the expert's rows its N = 16.
constexpr int64_t kDecodeMaxTokens = MOE_DECODE_MAX_TOKENS;

// Options that only the test build's entry points change; every product entry point passes
// the defaults. decode_hooks: the decode GEMM's scheduling fallbacks forced (bit 0: every
// first-unit guess wrong, bit 1: odd CTAs leave their offered unit to others);
// wait_limit_ns: the limit of every bounded wait in the GEMM kernels; withhold_release: the
// GEMM1 tiles of the first row tile (chained GEMMs) or of the first active expert (decode
// GEMMs) never publish their completion, so a GEMM2 wait runs out.
struct TestOptions {
  int32_t decode_hooks = 0;
  uint64_t wait_limit_ns = kWaitLimitNs;
  int32_t withhold_release = 0;
};

struct GemmLaunch {
  int mode;
  const uint8_t* a;      // [cap, K/2] packed rows in plan order
  const uint8_t* a_sf;   // [cap/128][Kp/64][512]
  const uint8_t* b;      // [El * Np, K/2]
  const uint8_t* b_sf;   // [El][Np/128][Kp/64][512]
  const float* alpha;    // [El]
  const float* alpha_gate;  // [El] gate scalars of a gated GEMM1 (else unused)
  const float* xs;       // per-token scale (GEMM1)
  const int32_t* padded_offsets;
  const int32_t* row_to_slot;
  int64_t cap, El, K, Kp, N, Np;
  int top_k, inter;
  bool gated;
  int act;
  float g2;
  void* out;
  uint8_t* out_sf;
  int32_t* dev_status;
  int32_t* tile_counter;
  // kG2Reduce: route weights (moe_weights_dtype_t storage) and routed scaling factor
  const void* route_w = nullptr;
  int route_w_dtype = 0;
  float rsf = 1.0f;
};

// GEMM1 (g1, kG1Fused) and GEMM2 (g2, kG2Rows or kG2Reduce) in one launch; mt_done holds
// cap / 128 zeroed counters
moe_status_t launch_gemm_chain(const GemmLaunch& g1, const GemmLaunch& g2, int32_t* mt_done, const TestOptions& topt,
                               cudaStream_t s);
// the same with the decode-shaped kernel (at most 16 rows per expert); e_done holds E_local
// zeroed counters
moe_status_t launch_gemm_decode(const GemmLaunch& g1, const GemmLaunch& g2, int32_t* e_done, int32_t* own,
                                const RoutingHint& hint, const TestOptions& topt, cudaStream_t s);
moe_status_t launch_permute(const int32_t* padded_offsets, int El, const int32_t* row_to_slot, int top_k,
                            int64_t cap, const uint8_t* xq, const uint8_t* xsf, int H, uint8_t* aq, uint8_t* asf,
                            int32_t* tile_counters, int32_t* mt_done, int64_t n_mt, const uint16_t* acc_init,
                            float* acc, int64_t acc_elems, cudaStream_t s);
// (mt_done: the row-tile and expert counters of one workspace, contiguous, n_mt ints)
moe_status_t launch_finalize(const uint16_t* rows, const void* topk_weights, int weights_dtype, float rsf,
                             const int32_t* token_to_row, int M, int top_k, int H, uint16_t* out, cudaStream_t s);
moe_status_t launch_store_acc(const float* acc, int64_t elems, uint16_t* out, cudaStream_t s);
// sizes, activation and expert count of a weights descriptor (api.cu)
moe_status_t check_weights(const moe_nvfp4_weights_t* w);
// permute (optional), GEMM1, GEMM2 and the combine of one validated forward (api.cu)
moe_status_t forward_chain(const int32_t* padded_offsets, const int32_t* row_to_slot, const int32_t* token_to_row,
                           int32_t M, int32_t top_k, const uint8_t* xq, const uint8_t* xsf, const float* xs,
                           const moe_nvfp4_weights_t* w, const void* prepared, const void* topk_weights,
                           int32_t topk_weights_dtype, float routed_scaling_factor, float fc2_input_scale,
                           int32_t do_finalize, uint16_t* out, uint16_t* gemm2_out, void* workspace,
                           int32_t* dev_status, void* const* step_events, int32_t num_step_events, bool run_permute,
                           const RoutingHint& hint, const TestOptions& topt, cudaStream_t s);
// The forward workspace carved into its buffers, and the prepared weights' parts (api.cu).
struct Bufs {
  int32_t* sched;
  int32_t* mtd;  // followed by the expert counters (edone)
  uint8_t *aq, *asf, *iq, *isf;
  uint16_t* g;
};
Bufs carve(void* ws, const WorkspaceLayout& L);
struct Prepared {
  const uint8_t *w1, *w1sf, *w2, *w2sf;
  const float *a1, *a2, *a1g;
};
Prepared prepared_ptrs(const void* prepared, const PreparedLayout& L);
// GEMM1 of a forward: the permuted activations times W1 into the intermediate (kG1Fused)
GemmLaunch gemm1_launch(const Dims& d, const WorkspaceLayout& L, const Bufs& b, const Prepared& pw,
                        const int32_t* padded_offsets, const int32_t* row_to_slot, const float* xs, int top_k,
                        int32_t* dev_status);
// moe_routed_forward with the test build's options (routed.cu)
moe_status_t routed_forward(const uint16_t* x, int32_t M, int64_t ld_x, int32_t act_scale_mode,
                            const int32_t* topk_ids, int32_t topk_ids_format, int32_t top_k, int32_t num_experts,
                            int32_t local_expert_offset, const void* topk_weights, int32_t topk_weights_dtype,
                            float routed_scaling_factor, const moe_nvfp4_weights_t* w, const void* prepared,
                            size_t prepared_bytes, float fc2_input_scale, int32_t do_finalize, uint16_t* out,
                            uint16_t* gemm2_out, int32_t* token_to_row, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* const* step_events, int32_t num_step_events,
                            const TestOptions& topt, moe_stream_t stream);
// the forward's argument checks shared with the test build's standalone GEMM1 (api.cu)
moe_status_t check_forward_common(const int32_t* padded_offsets, const int32_t* row_to_slot, int32_t M,
                                  int32_t top_k, const uint8_t* xq, const uint8_t* xsf, const float* xs,
                                  const moe_nvfp4_weights_t* w, const void* prepared, size_t prepared_bytes,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status, size_t ws_need);
moe_status_t launch_prepare_matrix(const uint8_t* src, const uint8_t* src_sf, int E, int rows, int rows_p, int K,
                                   int gated_inter, uint8_t* dst, uint8_t* dst_sf, cudaStream_t s);

}  // namespace moe

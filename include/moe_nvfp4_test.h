/*
 * moe_nvfp4_test.h - entry points of the TEST BUILD of the NVFP4 routed-MoE library
 * (libmoe_nvfp4_test.so). They are not part of the product ABI: the product library
 * (libmoe_nvfp4.so) exports none of them, keeps no hook or switch state, and runs every
 * kernel with the defaults below. The test library holds the same kernels and every
 * entry point of moe_nvfp4.h, plus these calls, which let tests reach paths that normal
 * inputs never take: a GEMM1 with plain epilogues, the decode GEMM's scheduling
 * fallbacks, and the bounded waits of the GEMM kernels running out.
 *
 * None of these calls keeps state between calls either: every option is an argument.
 */
#ifndef MOE_NVFP4_TEST_H_
#define MOE_NVFP4_TEST_H_

#include "moe_nvfp4.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Options of one test call. Zero-initialised options are NOT the defaults: start from
 * moe_test_default_options().
 *  decode_hooks      decode GEMM (batches of at most MOE_DECODE_MAX_TOKENS tokens, one-call
 *                    path): bit 0 makes every CTA's guess of its first unit's expert wrong (the
 *                    weight stages loaded before the dependency wait are reloaded); bit 1 makes
 *                    the odd CTAs leave their offered first unit to other CTAs. Results never
 *                    depend on either. Default 0.
 *  wait_limit_ns     limit of every bounded wait in the GEMM kernels (pipeline barriers, GEMM1
 *                    completion counters). Default 2 s.
 *  withhold_release  nonzero: the GEMM1 tiles of the first 128-row tile (chained GEMMs) or of
 *                    the first active expert (decode GEMMs) never publish their completion, so
 *                    the GEMM2 tiles that read them wait until wait_limit_ns runs out; the kernel
 *                    then ORs MOE_DEV_TIMEOUT into *dev_status and returns, with the outputs of
 *                    the abandoned tiles undefined. Default 0. */
typedef struct {
  int32_t decode_hooks;
  int32_t withhold_release;
  uint64_t wait_limit_ns;
} moe_test_options_t;

MOE_API moe_test_options_t moe_test_default_options(void);

/* moe_routed_forward with test options (NULL = the defaults, which is exactly
 * moe_routed_forward). */
MOE_API moe_status_t moe_test_routed_forward(const uint16_t* x, int32_t M, int64_t ld_x, int32_t act_scale_mode,
                                             const int32_t* topk_ids, int32_t topk_ids_format, int32_t top_k,
                                             int32_t num_experts, int32_t local_expert_offset,
                                             const void* topk_weights, int32_t topk_weights_dtype,
                                             float routed_scaling_factor, const moe_nvfp4_weights_t* w,
                                             const void* prepared, size_t prepared_bytes, float fc2_input_scale,
                                             int32_t do_finalize, uint16_t* out, uint16_t* gemm2_out,
                                             int32_t* token_to_row, void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, void* const* step_events,
                                             int32_t num_step_events, const moe_test_options_t* options,
                                             moe_stream_t stream);

/* The forward's permute and GEMM1 with a plain epilogue instead of the fused requantiser,
 * so tests can compare GEMM1 with the oracle before the activation and the requantiser.
 * mode 0: FP32 pre-activations y = acc * xs[t] * alpha1[e] (gate rows times the gate scalar)
 * into `dbg_out` [capacity, N1] (canonical [gate; up] column order); mode 1: the BF16
 * intermediate (after the activation) into `dbg_out` [capacity, I]. Real rows only.
 * Same arguments and workspace as moe_grouped_fp4_forward with MOE_OUTPUT_UNFINALIZED. */
MOE_API moe_status_t moe_test_gemm1(const int32_t* padded_offsets, const int32_t* row_to_slot, int32_t M,
                                    int32_t top_k, const uint8_t* xq, const uint8_t* xsf, const float* xs,
                                    const moe_nvfp4_weights_t* w, const void* prepared, size_t prepared_bytes,
                                    int32_t mode, void* dbg_out, void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_TEST_H_ */

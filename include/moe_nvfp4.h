/*
 * moe_nvfp4.h - C ABI of the NVFP4 routed-MoE expert path for GB300 (sm_103a).
 *
 * The path, in call order (one CUDA stream, no host synchronisation):
 *
 *   moe_quantize_input      BF16 hidden states -> NVFP4 activation pack
 *   moe_plan                routing ids -> expert-sorted plan (segments padded to 128 rows)
 *   moe_grouped_fp4_forward permute -> GEMM1 + activation + NVFP4 requant -> GEMM2
 *                           -> finalize (or the unfinalized rows)
 *   moe_finalize            ordered FP32 combine of unfinalized rows (standalone)
 *   moe_routed_forward      all of the above in one call, from BF16 hidden states
 *
 * plus one-time weight preparation (moe_quantize_weights, moe_prepare_weights).
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise, owned by
 *    the caller, and must be 16-byte aligned. The library never allocates device
 *    memory, never synchronises the stream and keeps no state between calls (one
 *    exception: the fixed scratch array of moe_plan_noalloc, below), so every call
 *    can be captured in a CUDA graph with fixed, capacity-sized buffers. Test hooks
 *    live in a separate test build (moe_nvfp4_test.h), not in this library.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns a status and launches nothing. A launch failure returns
 *    MOE_ERR_CUDA.
 *  - Data-dependent conditions found on the device are OR-ed into the caller's
 *    int32 `dev_status` word (MOE_DEV_* bits); no kernel traps. Zero it before
 *    the first call whose status you want to read.
 *  - BF16 tensors are passed as raw 16-bit storage (`uint16_t`), NVFP4 data as
 *    packed E2M1 bytes (two values per byte, the even logical element in the low
 *    nibble), block scales as float8_e4m3fn bytes, one per 16 consecutive values.
 *
 * Sources (web pages, cited by title and section):
 *  [CUDNN]  FlashInfer docs, flashinfer.fused_moe.CudnnGroupedGemmNvfp4Config
 *  [MCORE]  Megatron-Core API docs, core.inference.moe.flashinfer_nvfp4
 *  [ALPHA]  FlashInfer docs, flashinfer.fused_moe.alphamoe_nvfp4_aligned_moe
 *  [VLLM]   vLLM API docs, model_executor.layers.quantization.utils.flashinfer_utils
 *  [FROST]  FlashInfer docs, flashinfer.fused_moe.FrostLowLatencyConfig
 */
#ifndef MOE_NVFP4_H_
#define MOE_NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_NVFP4_ABI_VERSION 3

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef void* moe_stream_t; /* a cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARGUMENT = 1,  /* null pointer, negative size, bad enum */
  MOE_ERR_UNSUPPORTED_SHAPE = 2, /* H or I not a multiple of 128, too many experts, ... */
  MOE_ERR_MISALIGNED = 3,        /* a pointer or stride is not 16-byte aligned */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,
  MOE_ERR_CUDA = 5,              /* a CUDA call or launch failed */
  MOE_ERR_OVERLAP = 6            /* an output buffer overlaps an input */
} moe_status_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define MOE_DEV_DUPLICATE_EXPERT 1 /* a token names the same local expert twice ([CUDNN] "distinct experts") */
#define MOE_DEV_TIMEOUT 2          /* a bounded wait in a GEMM kernel gave up after 2 s; the kernel
                                      abandoned its remaining tiles and returned (outputs undefined) */

/* Expert activations. [MCORE] flashinfer_routed_nvfp4_moe(activation_type): squared-ReLU or
 * SwiGLU experts; [CUDNN] Activation functions: SwiGLU with default scalars, GeGLU, GELU, ReLU,
 * SiLU and Identity. Gated kinds (SwiGLU = silu(g)*u, GeGLU = gelu(g)*u) take W1 rows
 * [gate; up] (N1 = 2I); the others act on each of the I pre-activations (N1 = I).
 * GELU is x/2 * (1 + erf(x/sqrt(2))); SiLU is x / (1 + exp(-x)). */
typedef enum {
  MOE_ACT_SWIGLU = 0,
  MOE_ACT_RELU2 = 1,
  MOE_ACT_GEGLU = 2,
  MOE_ACT_GELU = 3,
  MOE_ACT_RELU = 4,
  MOE_ACT_SILU = 5,
  MOE_ACT_IDENTITY = 6
} moe_activation_t;

/* Storage of the route weights ([CUDNN] "Routing weights: packed, or unpacked FP32 / BF16").
 * MOE_WEIGHTS_PACKED: one int32 per slot holding the BF16 score in bits 31..16 and the
 * expert id, unsigned, in bits 15..0 (the pages name the packed form but not its bits; this
 * is the reading taken). [FROST]: "packed routing scores retain BF16 rounding". */
typedef enum { MOE_WEIGHTS_F32 = 0, MOE_WEIGHTS_BF16 = 1, MOE_WEIGHTS_PACKED = 2 } moe_weights_dtype_t;

/* Storage of the routing ids given to moe_plan: plain int32 ids, or the packed int32 slots
 * of MOE_WEIGHTS_PACKED (id = bits 15..0, so 0..65535; ids past the local range are masked). */
typedef enum { MOE_IDS_INT32 = 0, MOE_IDS_PACKED = 1 } moe_ids_format_t;

/* What moe_grouped_fp4_forward writes (its `do_finalize` argument).
 *  MOE_OUTPUT_UNFINALIZED  [CUDNN] MoEFinalizeConfig(do_finalize=False): BF16 expert rows
 *  MOE_OUTPUT_FINALIZED    ordered, deterministic FP32 combine into a fresh `out` ([FROST])
 *  MOE_OUTPUT_ACCUMULATE   [ALPHA]: contributions added in FP32 to the values already in
 *                          `out` (an FP32 copy of out is made first, out is rewritten once at
 *                          the end); the FP32 additions run in GEMM2's epilogue in whatever
 *                          order the tiles finish, so results may differ in the last bits
 *                          from run to run */
typedef enum {
  MOE_OUTPUT_UNFINALIZED = 0,
  MOE_OUTPUT_FINALIZED = 1,
  MOE_OUTPUT_ACCUMULATE = 2
} moe_output_mode_t;

/* Activation global scale: [CUDNN] "a global scale of one" (prepare_activations) or
 * [MCORE]/[VLLM] one FP32 decode scale per token computed online. */
typedef enum { MOE_SCALE_GLOBAL_ONE = 0, MOE_SCALE_PER_TOKEN = 1 } moe_act_scale_t;

/* Expert weights in the linear boundary layout of [ALPHA] (gemm1_weights / gemm2_weights):
 *   w1       [El, N1, H/2]  packed E2M1; N1 = 2*I rows [gate; up] for SwiGLU / GeGLU ([MCORE]
 *                            "MCore stores gated FC1 as [gate; up]"), N1 = I otherwise
 *   w1_sf    [El, N1, H/16] E4M3 block scales, row-major ("linear, contiguous")
 *   w1_alpha [El]           FP32 per-expert dequant (global decode scale) of W1
 *   w2       [El, H, I/2]   packed E2M1
 *   w2_sf    [El, H, I/16]  E4M3 block scales
 *   w2_alpha [El]           FP32 per-expert dequant of W2
 *   w1_gate_alpha [El]      optional FP32 per-expert dequant of the gate rows of a gated W1
 *                           ([ALPHA] output1_scale_gate_scalar, applied to each gate
 *                           accumulator before the activation, while w1_alpha plays
 *                           output1_scale_scalar for the up rows); NULL = w1_alpha for both.
 *                           Ignored by non-gated activations.
 * H and I must be multiples of 128 ([CUDNN] "hidden_size and intermediate_size must be
 * multiples of 128"); 1 <= El <= 512. moe_prepare_weights reads the pointers; the forward
 * reads only the sizes and `activation` (the prepared buffer is self-contained). */
typedef struct {
  const uint8_t* w1;
  const uint8_t* w1_sf;
  const float* w1_alpha;
  const uint8_t* w2;
  const uint8_t* w2_sf;
  const float* w2_alpha;
  int32_t num_local_experts;
  int32_t hidden;
  int32_t inter;
  int32_t activation; /* moe_activation_t */
  const float* w1_gate_alpha;
} moe_nvfp4_weights_t;

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char* moe_status_string(int32_t status);
MOE_API int32_t moe_abi_version(void);

/* ----------------------------------------------------------------------------------------
 * S1  moe_quantize_input - [CUDNN] Activations / prepare_activations; [MCORE]
 * quantize_routed_nvfp4_input; [VLLM] quantize_nvfp4_per_token_input.
 *   x   [M, ld_x] BF16 (first H columns used), ld_x >= H, ld_x % 8 == 0
 *   xq  [M, H/2]  packed E2M1 (out)
 *   xsf [M, H/16] E4M3 block scales, token-major linear (out)
 *   xs  [M]       FP32 decode scale per token (out): amax/2688 in MOE_SCALE_PER_TOKEN mode
 *                 (1 when the row is all zero), 1 in MOE_SCALE_GLOBAL_ONE mode.
 * Per 16-block, in IEEE float32: s = (max|x|/6) * g_enc; q = e4m3_rn_sat(s);
 * inv = q == 0 ? 0 : g_enc / q; code = e2m1_rn_sat(x * inv), with g_enc = 2688/amax
 * (per token) or 1. M == 0 is a no-op.
 * ---------------------------------------------------------------------------------------- */
MOE_API moe_status_t moe_quantize_input(const uint16_t* x, int32_t M, int32_t H, int64_t ld_x, int32_t mode,
                                uint8_t* xq, uint8_t* xsf, float* xs, moe_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * S2  moe_plan - [CUDNN] "rows and scale rows are permuted into expert order, each expert
 * segment padded to a multiple of 128 rows" (moe_sort); "assignments to non-local experts
 * are masked out"; [MCORE] "rows whose routing entries are -1 contribute zero";
 * [FROST] "expert IDs outside [0, num_experts) mark unrouted slots".
 *   topk_ids       [M, top_k] int32 global expert ids (topk_ids_format MOE_IDS_INT32), or the
 *                  packed slots of MOE_WEIGHTS_PACKED (MOE_IDS_PACKED: id = bits 15..0);
 *                  ids outside [local_expert_offset, local_expert_offset + El) are masked
 *                  (not errors)
 *   counts         [El]       routed rows per local expert (out)
 *   padded_offsets [El + 1]   segment starts, padded_offsets[l+1] - padded_offsets[l] =
 *                             roundup(counts[l], 128) (out)
 *   row_to_slot    [capacity] t*top_k + j of each real row, -1 for padding rows and for
 *                             every row from padded_offsets[El] to capacity (out)
 *   token_to_row   [M, top_k] row of slot (t, j) or -1 when masked (out)
 *   workspace      moe_plan_workspace_bytes(...) bytes of device scratch (may be NULL when 0)
 * Rows inside a segment are in ascending slot order (ascending token order). A token naming
 * one local expert twice sets MOE_DEV_DUPLICATE_EXPERT; the plan is still well defined.
 * ---------------------------------------------------------------------------------------- */
MOE_API size_t moe_plan_capacity(int32_t M, int32_t top_k, int32_t num_local_experts);
MOE_API size_t moe_plan_workspace_bytes(int32_t M, int32_t top_k, int32_t num_local_experts);
MOE_API moe_status_t moe_plan(const int32_t* topk_ids, int32_t topk_ids_format, int32_t M, int32_t top_k, int32_t num_experts,
                      int32_t local_expert_offset, int32_t num_local_experts, int32_t* counts,
                      int32_t* padded_offsets, int32_t* row_to_slot, int32_t* token_to_row,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      moe_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * moe_plan_noalloc - the pages have no counterpart of this call; it exists for callers of
 * this library that cannot allocate device memory: runtimes that hand out all device memory
 * from one pool reserved at start-up, C hosts with no device allocator, or code that must
 * not call cudaMalloc because it would synchronise the device mid-stream.
 * It computes exactly what moe_plan computes, with the same arguments minus the workspace:
 * the histogram scratch of the multi-block plan lives in a fixed array of
 * MOE_PLAN_NOALLOC_SCRATCH_BYTES of the library's own device memory, which every GPU that
 * loads the library holds until the process exits. The call allocates nothing.
 *  - Size limit: ceil(M * top_k / 2048) * num_local_experts * 4 bytes must not exceed
 *    MOE_PLAN_NOALLOC_SCRATCH_BYTES (inputs of at most 2048 slots need no scratch at all);
 *    larger inputs are rejected with MOE_ERR_UNSUPPORTED_SHAPE before anything runs.
 *  - The first call in each CUDA context looks up the array's device address in that
 *    context (cudaGetSymbolAddress) and caches it under the context's unique id, so a
 *    context torn down and re-created (cudaDeviceReset) is looked up afresh; make the first
 *    call in a context before any stream capture.
 *  - Every call on a device shares the one array and leaves its contents behind; nothing in
 *    it must start at zero, but calls that overlap on the GPU (other streams, other host
 *    threads) race on it and must be serialised by the caller.
 * ---------------------------------------------------------------------------------------- */
#define MOE_PLAN_NOALLOC_SCRATCH_BYTES (1 << 20)
MOE_API moe_status_t moe_plan_noalloc(const int32_t* topk_ids, int32_t topk_ids_format, int32_t M, int32_t top_k, int32_t num_experts,
                              int32_t local_expert_offset, int32_t num_local_experts, int32_t* counts,
                              int32_t* padded_offsets, int32_t* row_to_slot, int32_t* token_to_row,
                              int32_t* dev_status, moe_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Weight preparation (off the timed path).
 *
 * moe_quantize_weights - [MCORE] _global_encode_scale / _quantize_expert: one FP32 global
 * scale per expert matrix. Quantises `num_mats` BF16 matrices [rows, cols] (contiguous) to
 * data [num_mats, rows, cols/2], sf [num_mats, rows, cols/16] (linear) and alpha
 * [num_mats] = amax/2688 (1 for an all-zero matrix), with g_enc = 2688/amax in the block
 * rule of moe_quantize_input. `amax_scratch` holds num_mats floats of device scratch.
 *
 * moe_prepare_weights - lays the linear weights out for the kernels (w1_gate_alpha, or w1_alpha
 * when it is NULL, is copied into the buffer as the gate scalars): SwiGLU gate and up rows
 * interleaved in 128-row blocks (so one 256-row GEMM1 tile holds matching gate and up
 * columns), rows padded to 256 per expert, block scales in 128-row x 4-scale tiles.
 * The buffer (moe_prepared_weights_bytes) is self-contained; refreshing it in place keeps
 * captured addresses valid ([MCORE] prepare_routed_nvfp4_weights(out=...)).
 * ---------------------------------------------------------------------------------------- */
MOE_API moe_status_t moe_quantize_weights(const uint16_t* w, int32_t num_mats, int32_t rows, int32_t cols,
                                  uint8_t* data, uint8_t* sf, float* alpha, float* amax_scratch,
                                  moe_stream_t stream);
MOE_API size_t moe_prepared_weights_bytes(const moe_nvfp4_weights_t* w);
MOE_API moe_status_t moe_prepare_weights(const moe_nvfp4_weights_t* w, void* prepared, size_t prepared_bytes,
                                 moe_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * S3-S8  moe_grouped_fp4_forward - [CUDNN] Pipeline: permutation, GEMM1 (rows x expert
 * global dequant), typed activation, NVFP4 requant of the BF16 intermediate "straight into
 * [GEMM2's] layout", GEMM2, finalize; MoEFinalizeConfig(do_finalize=False) returns
 * [gemm2_out, expert_weights, token_to_row]. [ALPHA] tensor contract and 16-byte alignment.
 *   padded_offsets, row_to_slot, token_to_row  from moe_plan
 *   xq, xsf, xs        activation pack from moe_quantize_input ([M, H/2], [M, H/16], [M])
 *   w, prepared        sizes/activation and the moe_prepare_weights buffer
 *   topk_weights       [M, top_k] route weights, FP32, BF16 or packed per topk_weights_dtype
 *                      (entries of masked slots are never read)
 *   routed_scaling_factor  finite FP32 scalar applied to each routed contribution ([ALPHA]
 *                      routed_scaling_factor): the combine uses w' = fp32(w * factor); 1.0 = none
 *   fc2_input_scale    static FP32 encode scale of the intermediate (1.0 = global scale one);
 *                      GEMM2 rows are multiplied by alpha2[e] / fc2_input_scale
 *   do_finalize (moe_output_mode_t):
 *     MOE_OUTPUT_FINALIZED    out [M, H] BF16 = bf16(sum_j w'[t,j] * gemm2 row), ordered FP32
 *                      multiply + add over ascending j ([FROST] ordered combine); gemm2_out
 *                      may be NULL (rows go to the workspace)
 *     MOE_OUTPUT_UNFINALIZED  gemm2_out [capacity, H] BF16 expert outputs, bf16(y2) in real
 *                      rows, padding rows untouched; out may be NULL
 *     MOE_OUTPUT_ACCUMULATE   out [M, H] BF16 (read and written) = bf16(out + sum_j y2 * w'[t,j])
 *                      with y2 the FP32 GEMM2 row (not rounded to BF16), FP32 additions in
 *                      any order ([ALPHA]: accumulation in an FP32 [M, H] buffer initialised
 *                      from out, converted back once); rows of tokens with no local slot keep
 *                      their value; gemm2_out may be NULL
 *   workspace          moe_forward_workspace_bytes(...) bytes of device scratch
 *   step_events        optional array of `num_step_events` (0 or 5) cudaEvent_t recorded on
 *                      `stream` before permute, gemm1, gemm2, finalize and at the end. GEMM1
 *                      and GEMM2 run as one chained launch (the GEMM2 tiles of a 128-row tile
 *                      start as soon as its GEMM1 tiles are written), whose time falls
 *                      between the gemm1 and gemm2 marks
 * ---------------------------------------------------------------------------------------- */
/* Batches of at most this many tokens run GEMM1 and GEMM2 with the operands swapped
 * (the weight tile as the MMA's 128-row operand, each expert's token rows as its 16
 * columns). A token naming one expert twice (MOE_DEV_DUPLICATE_EXPERT) can give an expert
 * more than 16 rows; rows past the 16th are then not computed. */
#define MOE_DECODE_MAX_TOKENS 16
MOE_API size_t moe_forward_workspace_bytes(int32_t M, int32_t top_k, const moe_nvfp4_weights_t* w,
                                   int32_t do_finalize);
/* Byte offsets inside the forward workspace of: [0] permuted activations [cap, H/2],
 * [1] their scales (128x4 tiles), [2] intermediate [cap, I/2], [3] its scales,
 * [4] gemm2 rows [cap, H] BF16 (MOE_OUTPUT_FINALIZED) or the FP32 accumulator [M, H]
 * (MOE_OUTPUT_ACCUMULATE), 0 otherwise, [5] total. For tests and tools. */
MOE_API moe_status_t moe_forward_workspace_layout(int32_t M, int32_t top_k, const moe_nvfp4_weights_t* w,
                                          int32_t do_finalize, size_t offsets[6]);
MOE_API moe_status_t moe_grouped_fp4_forward(const int32_t* padded_offsets, const int32_t* row_to_slot,
                                     const int32_t* token_to_row, int32_t M, int32_t top_k,
                                     const uint8_t* xq, const uint8_t* xsf, const float* xs,
                                     const moe_nvfp4_weights_t* w, const void* prepared,
                                     size_t prepared_bytes, const void* topk_weights,
                                     int32_t topk_weights_dtype, float routed_scaling_factor,
                                     float fc2_input_scale, int32_t do_finalize, uint16_t* out,
                                     uint16_t* gemm2_out, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, void* const* step_events,
                                     int32_t num_step_events, moe_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * S7  moe_finalize - [CUDNN] moe_unpermute; [FROST] "ordered, separate FP32 multiplication
 * and addition"; unrouted slots and their scores are ignored.
 *   gemm2_out    [rows, H] BF16 expert rows
 *   topk_weights [M, top_k] route weights, FP32, BF16 or packed (topk_weights_dtype)
 *   routed_scaling_factor  finite FP32 scalar, w' = fp32(w * factor) ([ALPHA])
 *   token_to_row [M, top_k] row per slot or -1;  out [M, H] BF16
 * out[t,:] = bf16(acc) with acc = 0; acc = acc + w'[t,j]*row for j = 0..top_k-1, row != -1.
 * A token with every slot masked gets a zero row.
 * ---------------------------------------------------------------------------------------- */
MOE_API moe_status_t moe_finalize(const uint16_t* gemm2_out, const void* topk_weights,
                          int32_t topk_weights_dtype, float routed_scaling_factor,
                          const int32_t* token_to_row, int32_t M, int32_t top_k, int32_t H,
                          uint16_t* out, moe_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * moe_routed_forward - the whole layer in one call ([MCORE] flashinfer_routed_nvfp4_moe:
 * BF16 hidden states, routing map and probabilities in, the layer output out). It computes
 * exactly what moe_quantize_input, moe_plan and moe_grouped_fp4_forward compute in sequence
 * (bit for bit, except the order of the FP32 additions of MOE_OUTPUT_ACCUMULATE). For small
 * batches (M * top_k <= 2048 and M * H <= 131072) the quantiser, the plan and the
 * permutation run as one kernel.
 *   x             [M, ld_x] BF16 hidden states (first H columns used), ld_x >= H, ld_x % 8 == 0
 *   act_scale_mode  moe_act_scale_t, as moe_quantize_input
 *   topk_ids, topk_ids_format, num_experts, local_expert_offset  as moe_plan
 *   topk_weights, topk_weights_dtype, routed_scaling_factor, w, prepared, fc2_input_scale,
 *   do_finalize, out, gemm2_out  as moe_grouped_fp4_forward (packed slots may pass the same
 *                 buffer as topk_ids and topk_weights)
 *   token_to_row  [M, top_k] int32 (out): the plan row of each slot or -1 (the third element of
 *                 the unfinalized result)
 *   workspace     moe_routed_forward_workspace_bytes(M, top_k, w, do_finalize) bytes; it holds
 *                 the activation pack, the plan and the forward workspace
 *   step_events   0 or 5 cudaEvent_t recorded before the prologue (quantise, plan, permute),
 *                 GEMM1, GEMM2, the combine, and at the end
 * Outputs must not overlap any input, the workspace or each other (MOE_ERR_OVERLAP).
 * Host buffers: x, topk_ids, topk_weights and, with do_finalize = MOE_OUTPUT_FINALIZED, out
 * may instead be page-locked host memory that the device addresses directly (cudaHostAlloc
 * or cudaHostRegister, unified addressing). The kernels then read and write them in place
 * over the CPU-GPU link, with plain loads and stores. For small batches this saves the fixed
 * latency of separate copies. For large ones the copy engine moves the data faster.
 * ---------------------------------------------------------------------------------------- */
MOE_API size_t moe_routed_forward_workspace_bytes(int32_t M, int32_t top_k, const moe_nvfp4_weights_t* w,
                                                  int32_t do_finalize);
MOE_API moe_status_t moe_routed_forward(const uint16_t* x, int32_t M, int64_t ld_x, int32_t act_scale_mode,
                                        const int32_t* topk_ids, int32_t topk_ids_format, int32_t top_k,
                                        int32_t num_experts, int32_t local_expert_offset,
                                        const void* topk_weights, int32_t topk_weights_dtype,
                                        float routed_scaling_factor, const moe_nvfp4_weights_t* w,
                                        const void* prepared, size_t prepared_bytes, float fc2_input_scale,
                                        int32_t do_finalize, uint16_t* out, uint16_t* gemm2_out,
                                        int32_t* token_to_row, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_status, void* const* step_events, int32_t num_step_events,
                                        moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H_ */

// The whole layer in one call: BF16 hidden states and routing in, the combined BF16 output
// (or the unfinalized rows) out.
//
// Sources: Megatron-Core core.inference.moe.flashinfer_nvfp4 (flashinfer_routed_nvfp4_moe:
// hidden states, routing map and probabilities in, the layer output out;
// quantize_routed_nvfp4_input); FlashInfer flashinfer.fused_moe.CudnnGroupedGemmNvfp4Config
// (Pipeline: NVFP4 activation pack, expert-sorted permutation, GEMM1, typed activation,
// GEMM2, finalize).
//
// Small batches (decode: at most 2048 routed slots and 2^17 hidden values) run the
// quantiser, the plan and the permutation in one kernel (one CTA per token group, each
// building the small plan itself), and GEMM1 and GEMM2 as one launch, so the step is
// three launches (prologue, GEMMs, combine)
// instead of six; each of those steps is latency-bound at these sizes. Larger batches run the separate kernels of
// moe_plan, a quantiser that stores straight into the plan rows, and the GEMMs and combine
// of moe_grouped_fp4_forward. Both paths compute the same bytes as the separate calls: the
// quantisers and the plan follow the same arithmetic and order as the separate kernels.
#include <math.h>

#include "common.cuh"
#include "host_util.h"
#include "layout.h"
#include "plan_device.cuh"

namespace moe {
namespace {

constexpr int kPrologueThreads = kPlanThreads;               // 1024
constexpr int64_t kPrologueMaxSlots = kSlotsPerBlock;        // the one-block plan
constexpr int64_t kPrologueMaxValues = int64_t(1) << 17;     // M * H

// Routed-call workspace: activation pack, plan arrays and scratch, then the forward workspace.
struct RoutedLayout {
  size_t xq, xsf, xs, counts, padded, r2s, plan_ws, fwd, total;
  int64_t cap;
};

RoutedLayout routed_layout(const Dims& d, int64_t M, int64_t k, int out_mode) {
  RoutedLayout R;
  size_t c = 0;
  R.cap = plan_capacity_rows(M, k, d.El);
  R.xq = take(c, M * d.H / 2);
  R.xsf = take(c, M * d.H / 16);
  R.xs = take(c, M * 4);
  R.counts = take(c, d.El * 4);
  R.padded = take(c, (d.El + 1) * 4);
  R.r2s = take(c, (R.cap > 0 ? R.cap : 1) * 4);
  R.plan_ws = take(c, moe_plan_workspace_bytes(static_cast<int32_t>(M), static_cast<int32_t>(k),
                                               static_cast<int32_t>(d.El)));
  R.fwd = take(c, workspace_layout(d, M, k, out_mode).total);
  R.total = c;
  return R;
}

bool small_batch(int64_t M, int64_t k, int64_t H) {
  return M * k <= kPrologueMaxSlots && M * H <= kPrologueMaxValues;
}

constexpr int kPrologueMaxRows = static_cast<int>(kPrologueMaxValues / 128);  // H >= 128
constexpr int kPrologueMaxCtas = 32;
constexpr int kPrologueStageBlocks = 1024;  // own 16-value blocks quantised during the plan scan

// A grid of G <= 32 CTAs, CTA c taking tokens c, c + G, ... Every CTA builds the whole plan
// in shared memory (at most 2048 slots: the one-block plan of plan_single_kernel, from the
// routing ids alone), so no CTA waits for another:
//  (0) the routed-slot histogram and, for per-token scales, its tokens' max |x| (thread per
//      16-value block, maximum through shared memory);
//  (1) the plan, written out in shares: CTA 0 the counts and padded offsets, CTA c the
//      padding rows of experts c, c + G, ... and token_to_row / row_to_slot of its own
//      tokens' slots (with the duplicate-expert check); each CTA zeroes a slice of the GEMM
//      counters;
//  (2) NVFP4 quantisation of its tokens' 16-value blocks (the arithmetic of
//      quantize_rows_kernel), each block's 8 code bytes and scale byte stored straight into
//      every plan row of the token (the permuted operand of GEMM1 and its 128x4 scale
//      tiles): the quantised activations never make a round trip through memory. When the
//      own blocks fit in shared memory they are quantised while warp 0 scans the plan, and
//      only stored once the rows are placed.
// Also its tokens' scales and, for an accumulated output, the FP32 copy of their rows of out.
__global__ void __launch_bounds__(kPrologueThreads) small_prologue_kernel(
    const uint16_t* __restrict__ x, int M, int H, int64_t ld, int per_token, const int32_t* __restrict__ ids,
    int id_mask, int top_k, int off, int El, float* __restrict__ xs, int32_t* __restrict__ counts,
    int32_t* __restrict__ padded_offsets, int32_t* row_to_slot, int32_t* token_to_row, int32_t* dev_status,
    uint8_t* __restrict__ aq, uint8_t* __restrict__ asf, int32_t* __restrict__ tile_counters,
    int32_t* __restrict__ mt_done, int n_mt, const uint16_t* __restrict__ acc_init, float* __restrict__ acc) {
  __shared__ PlanSmem sm;
  __shared__ unsigned s_amax[kPrologueMaxRows];      // max |x| of each own token (bits of a non-negative float)
  __shared__ int32_t s_row[kPrologueMaxSlots];       // plan row of each slot
  __shared__ __align__(16) uint2 s_code[kPrologueStageBlocks];    // own blocks' codes (when they fit)
  __shared__ __align__(16) uint8_t s_qsc[kPrologueStageBlocks];   // and scale bytes
  __shared__ int16_t s_loc[kPrologueMaxSlots];       // local expert of each slot, or -1
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const bool lead = c == 0;
  const int n_own = (M - c + G - 1) / G;             // own tokens c + i*G, i < n_own
  zero_tables(sm, El);
  for (int i = threadIdx.x; i < n_own; i += kPrologueThreads) s_amax[i] = 0u;
  pdl_wait();
  // after the wait: the GEMM launched early reads the routing ids and the weights before its
  // own wait, and finds every kernel before this one done
  pdl_trigger();
  if (lead && threadIdx.x < 2) tile_counters[threadIdx.x] = 0;
  for (int i = c * kPrologueThreads + threadIdx.x; i < n_mt; i += G * kPrologueThreads) mt_done[i] = 0;
  const int n = M * top_k;
  const int nblk = H / kBlock;
  const int nb_own = n_own * nblk;
  __syncthreads();
  // (0) histogram of the routed slots per local expert; own tokens' maxima
  for (int s = threadIdx.x; s < n; s += kPrologueThreads) {
    const int l = local_of(entry_id(ids, s, id_mask), off, El);
    s_loc[s] = static_cast<int16_t>(l);
    if (l >= 0) atomicAdd(&sm.cnt[l], 1);
  }
  if (per_token) {
    for (int bi = threadIdx.x; bi < nb_own; bi += kPrologueThreads) {
      const int i = bi / nblk, b = bi - i * nblk;
      float v[16];
      load_block16(x + static_cast<int64_t>(c + i * G) * ld + b * kBlock, v);
      float amax = 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
      atomicMax(&s_amax[i], __float_as_uint(amax));
    }
  }
  __syncthreads();
  // (1) plan: warp 0 scans the expert counts while the other warps quantise the own blocks
  const bool staged = nb_own <= kPrologueStageBlocks;
  if (threadIdx.x < 32) {
    scan_padded(sm, El);
  } else if (staged) {
    for (int bi = threadIdx.x - 32; bi < nb_own; bi += kPrologueThreads - 32) {
      const int i = bi / nblk, b = bi - i * nblk;
      float g = 1.0f;
      if (per_token) {
        const float amax = __uint_as_float(s_amax[i]);
        if (amax > 0.0f) g = __fdiv_rn(kGlobalNumerator, amax);
      }
      float v[16];
      load_block16(x + static_cast<int64_t>(c + i * G) * ld + b * kBlock, v);
      uint32_t codes[2];
      s_qsc[bi] = static_cast<uint8_t>(quantize_block16(v, g, codes));
      s_code[bi] = make_uint2(codes[0], codes[1]);
    }
  }
  __syncthreads();
  if (lead)
    for (int l = threadIdx.x; l <= El; l += kPrologueThreads) {
      padded_offsets[l] = sm.cursor[l];
      if (l < El) counts[l] = sm.cnt[l];
    }
  // -1 on the padding rows of experts c, c + G, ... (one warp per expert); rows past the
  // padded total are never read by the GEMMs, so (unlike moe_plan's output) this internal
  // row_to_slot leaves them unwritten
  {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int l = c + warp * G; l < El; l += G * (kPrologueThreads / 32)) {
      const int b = sm.cursor[l] + sm.cnt[l];
      const int e = sm.cursor[l] + (sm.cnt[l] + kSegAlign - 1) / kSegAlign * kSegAlign;
      for (int r = b + lane; r < e; r += 32) row_to_slot[r] = -1;
    }
  }
  __syncthreads();
  place_range(ids, id_mask, 0, n, top_k, off, El, sm, nullptr, s_row, nullptr);
  __syncthreads();
  // own tokens' slots: token_to_row, row_to_slot and the duplicate-expert check (as moe_plan:
  // a routed slot naming the same expert as an earlier slot of its token; for local slots
  // equal ids are equal local indices, kept in shared memory since the histogram)
  for (int it = threadIdx.x; it < n_own * top_k; it += kPrologueThreads) {
    const int i = it / top_k, j = it - i * top_k;
    const int sl = (c + i * G) * top_k + j;
    const int row = s_row[sl];
    token_to_row[sl] = row;
    if (row >= 0) {
      row_to_slot[row] = sl;
      const int l = s_loc[sl];
      for (int q = sl - j; q < sl; ++q)
        if (s_loc[q] == l) atomicOr(dev_status, MOE_DEV_DUPLICATE_EXPERT);
    }
  }
  const int kcols_p = static_cast<int>(roundup64(H, kTileK) / 16);  // scale columns incl. K padding
  if (staged) {
    // (2) the staged blocks into every plan row of their token: per row 16-byte code vectors
    // (two blocks) and 4-byte scale groups (the four scales of a 128x4 tile row are
    // contiguous), zero groups on the K padding; H is a multiple of 128, so the blocks split
    // evenly into both
    const int nv = nblk / 2, ng = kcols_p / 4, per_row = nv + ng;
    const uint4* c16 = reinterpret_cast<const uint4*>(s_code);
    const uint32_t* q4 = reinterpret_cast<const uint32_t*>(s_qsc);
    for (int it = threadIdx.x; it < n_own * top_k * per_row; it += kPrologueThreads) {
      const int sl = it / per_row, w = it - sl * per_row;  // own slot: token i, slot j
      const int i = sl / top_k, j = sl - i * top_k;
      const int row = s_row[(c + i * G) * top_k + j];
      if (row < 0) continue;
      if (w < nv) {
        reinterpret_cast<uint4*>(aq + static_cast<int64_t>(row) * (H / 2))[w] = c16[i * nv + w];
      } else {
        const int g = w - nv;
        *reinterpret_cast<uint32_t*>(asf + sf_tile_offset(row, 4 * g, kcols_p)) = g < nblk / 4 ? q4[i * (nblk / 4) + g] : 0u;
      }
    }
    for (int i = threadIdx.x; i < n_own; i += kPrologueThreads) {
      float dec = 1.0f;
      if (per_token) {
        const float amax = __uint_as_float(s_amax[i]);
        if (amax > 0.0f) dec = __fdiv_rn(amax, kGlobalNumerator);
      }
      xs[c + i * G] = dec;
    }
  } else {
    // (2) own tokens: one thread per (token, slot, block), consecutive threads on consecutive
    // blocks of one plan row; each block is quantised by the same arithmetic for every slot
    const int per_tok = top_k * nblk;
    for (int it = threadIdx.x; it < n_own * per_tok; it += kPrologueThreads) {
      const int i = it / per_tok, rem = it - i * per_tok;
      const int j = rem / nblk, b = rem - j * nblk;
      const int r = c + i * G;
      const int row = s_row[r * top_k + j];
      if (row < 0 && !(j == 0 && b == 0)) continue;
      float g = 1.0f, dec = 1.0f;
      if (per_token) {
        const float amax = __uint_as_float(s_amax[i]);
        if (amax > 0.0f) {
          g = __fdiv_rn(kGlobalNumerator, amax);
          dec = __fdiv_rn(amax, kGlobalNumerator);
        }
      }
      if (j == 0 && b == 0) xs[r] = dec;
      if (row < 0) continue;
      float v[16];
      load_block16(x + static_cast<int64_t>(r) * ld + b * kBlock, v);
      uint32_t codes[2];
      const uint32_t q = quantize_block16(v, g, codes);
      *reinterpret_cast<uint2*>(aq + static_cast<int64_t>(row) * (H / 2) + b * 8) = make_uint2(codes[0], codes[1]);
      asf[sf_tile_offset(row, b, kcols_p)] = static_cast<uint8_t>(q);
    }
    // zero scales on the K padding columns of the own tokens' routed rows (H not a multiple of 256)
    const int npad = kcols_p - nblk;
    for (int it = threadIdx.x; it < n_own * top_k * npad; it += kPrologueThreads) {
      const int sl = it / npad;                         // own slot index: token i, slot j
      const int i = sl / top_k, j = sl - i * top_k;
      const int row = s_row[(c + i * G) * top_k + j];
      if (row >= 0) asf[sf_tile_offset(row, nblk + (it - sl * npad), kcols_p)] = 0;
    }
  }
  // accumulated output: acc = fp32(out) on the own tokens' rows
  if (acc != nullptr) {
    const int h8 = H / 8;
    for (int it = threadIdx.x; it < n_own * h8; it += kPrologueThreads) {
      const int i = it / h8;
      const int64_t e = static_cast<int64_t>(c + i * G) * h8 + (it - i * h8);
      const uint4 v = reinterpret_cast<const uint4*>(acc_init)[e];
      float4* d = reinterpret_cast<float4*>(acc) + 2 * e;
      d[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                         __uint_as_float(v.y & 0xFFFF0000u));
      d[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u), __uint_as_float(v.w << 16),
                         __uint_as_float(v.w & 0xFFFF0000u));
    }
  }
}

// Larger batches: one warp per token computes its scale (per-token max |x| over the row,
// then the row is read again from L1/L2) and quantises each 16-value block once (the
// arithmetic of quantize_rows_kernel) into the warp's shared-memory buffer; after the plan it
// stores each block's codes and scale straight into every plan row of the token, so the
// quantised activations are never written token-major and read back by a permutation. The
// first token of every warp is read and quantised before the dependency wait (x is an
// input of the step, and the plan's first kernel lets its dependents start only once every
// earlier kernel is done), so that work overlaps the plan. Block 0 zeroes the GEMM counters;
// an accumulated output's FP32 copy of out is made by all threads.
// Dynamic shared memory: (warps per block) x (H/16) x 9 bytes.
__global__ void __launch_bounds__(256) quantize_scatter_kernel(
    const uint16_t* __restrict__ x, int M, int H, int64_t ld, int per_token, int top_k,
    const int32_t* __restrict__ token_to_row, float* __restrict__ xs, uint8_t* __restrict__ aq,
    uint8_t* __restrict__ asf, int32_t* __restrict__ counters, int n_counters, const uint16_t* __restrict__ acc_init,
    float* __restrict__ acc) {
  extern __shared__ uint8_t qs_smem[];
  pdl_trigger();
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int nblk = H / kBlock;
  const int kcols_p = static_cast<int>(roundup64(H, kTileK) / 16);
  uint2* s_codes = reinterpret_cast<uint2*>(qs_smem) + static_cast<int64_t>(wib) * nblk;
  uint8_t* s_q = qs_smem + static_cast<int64_t>(blockDim.x >> 5) * nblk * 8 + static_cast<int64_t>(wib) * nblk;
  // the token's scale and quantised blocks into the warp's buffers; returns the decode scale
  auto stage = [&](int64_t t) -> float {
    const uint16_t* row = x + t * ld;
    float g = 1.0f, dec = 1.0f;
    if (per_token) {
      float amax = 0.0f;
      for (int b = lane; b < nblk; b += 32) {
        float v[16];
        load_block16(row + b * kBlock, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
      }
      amax = warp_max(amax);
      if (amax > 0.0f) {
        g = __fdiv_rn(kGlobalNumerator, amax);
        dec = __fdiv_rn(amax, kGlobalNumerator);
      }
    }
    for (int b = lane; b < nblk; b += 32) {
      float v[16];
      load_block16(row + b * kBlock, v);
      uint32_t codes[2];
      s_q[b] = static_cast<uint8_t>(quantize_block16(v, g, codes));
      s_codes[b] = make_uint2(codes[0], codes[1]);
    }
    return dec;
  };
  float dec = warp0 < M ? stage(warp0) : 0.0f;
  pdl_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
  for (int64_t t = warp0; t < M; t += nwarps) {
    if (t != warp0) dec = stage(t);
    __syncwarp();  // the staged blocks are read by other lanes below
    // the token's plan rows (lane j holds slot j's row): per row, 16-byte code vectors (two
    // blocks) and 4-byte scale groups (the four scales of a 128x4 tile row are contiguous);
    // H is a multiple of 128, so the blocks split evenly into both
    const int my_row = lane < top_k ? token_to_row[t * top_k + lane] : -1;
    const uint4* c16 = reinterpret_cast<const uint4*>(s_codes);
    const uint32_t* q4 = reinterpret_cast<const uint32_t*>(s_q);
    for (int j = 0; j < top_k; ++j) {
      const int prow = j < 32 ? __shfl_sync(0xffffffffu, my_row, j) : token_to_row[t * top_k + j];
      if (prow < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(aq + static_cast<int64_t>(prow) * (H / 2));
      for (int v = lane; v < nblk / 2; v += 32) dst[v] = c16[v];
      // scale groups, then zero groups on the K padding (H not a multiple of 256)
      for (int g = lane; g < kcols_p / 4; g += 32)
        *reinterpret_cast<uint32_t*>(asf + sf_tile_offset(prow, 4 * g, kcols_p)) = g < nblk / 4 ? q4[g] : 0u;
    }
    __syncwarp();  // every lane's reads of the buffers precede the next token's staging
    if (lane == 0) xs[t] = dec;
  }
  if (acc != nullptr) {
    const int64_t n8 = static_cast<int64_t>(M) * H / 8;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += nth) {
      const uint4 v = reinterpret_cast<const uint4*>(acc_init)[i];
      float4* d = reinterpret_cast<float4*>(acc) + 2 * i;
      d[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                         __uint_as_float(v.y & 0xFFFF0000u));
      d[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u), __uint_as_float(v.w << 16),
                         __uint_as_float(v.w & 0xFFFF0000u));
    }
  }
}

moe_status_t record_mark(void* ev, cudaStream_t s) {
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  MOE_CUDA(cudaStreamIsCapturing(s, &capturing));
  if (capturing == cudaStreamCaptureStatusActive)
    MOE_CUDA(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal));
  else
    MOE_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(ev), s));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_routed_forward_workspace_bytes(int32_t M, int32_t top_k, const moe_nvfp4_weights_t* w,
                                                     int32_t do_finalize) {
  if (check_weights(w) != MOE_OK || M < 0 || top_k < 1) return 0;
  if (do_finalize < MOE_OUTPUT_UNFINALIZED || do_finalize > MOE_OUTPUT_ACCUMULATE) return 0;
  return routed_layout(make_dims(w), M, top_k, do_finalize).total;
}

moe_status_t moe::routed_forward(const uint16_t* x, int32_t M, int64_t ld_x, int32_t act_scale_mode,
                                 const int32_t* topk_ids, int32_t topk_ids_format, int32_t top_k, int32_t num_experts,
                                 int32_t local_expert_offset, const void* topk_weights, int32_t topk_weights_dtype,
                                 float routed_scaling_factor, const moe_nvfp4_weights_t* w, const void* prepared,
                                 size_t prepared_bytes, float fc2_input_scale, int32_t do_finalize, uint16_t* out,
                                 uint16_t* gemm2_out, int32_t* token_to_row, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* const* step_events, int32_t num_step_events,
                                 const TestOptions& topt, moe_stream_t stream) {
  moe_status_t st = check_weights(w);
  if (st != MOE_OK) return st;
  MOE_CHECK(M >= 0 && top_k >= 1, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(do_finalize >= MOE_OUTPUT_UNFINALIZED && do_finalize <= MOE_OUTPUT_ACCUMULATE, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(act_scale_mode == MOE_SCALE_GLOBAL_ONE || act_scale_mode == MOE_SCALE_PER_TOKEN,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(topk_ids_format == MOE_IDS_INT32 || topk_ids_format == MOE_IDS_PACKED, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(topk_weights_dtype >= MOE_WEIGHTS_F32 && topk_weights_dtype <= MOE_WEIGHTS_PACKED,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(isfinite(routed_scaling_factor) && isfinite(fc2_input_scale) && fc2_input_scale > 0.0f,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(num_step_events == 0 || (num_step_events == 5 && step_events != nullptr), MOE_ERR_INVALID_ARGUMENT);
  const Dims d = make_dims(w);
  MOE_CHECK(num_experts >= 1 && local_expert_offset >= 0 && local_expert_offset + d.El <= num_experts,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(ld_x >= d.H && ld_x % 8 == 0, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(static_cast<int64_t>(M) * top_k < (int64_t(1) << 30), MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(prepared != nullptr && prepared_bytes >= prepared_layout(d).total, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(prepared), MOE_ERR_MISALIGNED);
  const RoutedLayout R = routed_layout(d, M, top_k, do_finalize);
  MOE_CHECK(workspace_bytes >= R.total, MOE_ERR_WORKSPACE_TOO_SMALL);
  if (M == 0) return MOE_OK;
  const bool finalized = do_finalize != MOE_OUTPUT_UNFINALIZED;
  MOE_CHECK(x && topk_ids && topk_weights && token_to_row && workspace && dev_status, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(finalized ? out != nullptr : gemm2_out != nullptr, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(x) && aligned16(topk_ids) && aligned16(topk_weights) && aligned16(token_to_row) &&
                aligned16(workspace) && aligned16(dev_status) && aligned16(finalized ? out : gemm2_out),
            MOE_ERR_MISALIGNED);
  const size_t xb = static_cast<size_t>(M - 1) * ld_x * 2 + d.H * 2;
  const size_t ib = static_cast<size_t>(M) * top_k * 4;
  const size_t wb = static_cast<size_t>(M) * top_k * (topk_weights_dtype == MOE_WEIGHTS_BF16 ? 2 : 4);
  const size_t pb = prepared_bytes;
  // outputs overlap no input and no other output
  void* const o = finalized ? static_cast<void*>(out) : static_cast<void*>(gemm2_out);
  const size_t ob = finalized ? static_cast<size_t>(M) * d.H * 2 : static_cast<size_t>(R.cap) * d.H * 2;
  MOE_CHECK(!overlaps(o, ob, x, xb) && !overlaps(o, ob, topk_ids, ib) && !overlaps(o, ob, topk_weights, wb) &&
                !overlaps(o, ob, token_to_row, ib) && !overlaps(o, ob, workspace, R.total) &&
                !overlaps(o, ob, prepared, pb),
            MOE_ERR_OVERLAP);
  MOE_CHECK(!overlaps(token_to_row, ib, x, xb) && !overlaps(token_to_row, ib, topk_ids, ib) &&
                !overlaps(token_to_row, ib, topk_weights, wb) && !overlaps(token_to_row, ib, workspace, R.total) &&
                !overlaps(token_to_row, ib, prepared, pb),
            MOE_ERR_OVERLAP);
  MOE_CHECK(!overlaps(workspace, R.total, x, xb) && !overlaps(workspace, R.total, topk_ids, ib) &&
                !overlaps(workspace, R.total, topk_weights, wb) && !overlaps(workspace, R.total, prepared, pb),
            MOE_ERR_OVERLAP);

  cudaStream_t s = as_stream(stream);
  uint8_t* b = static_cast<uint8_t*>(workspace);
  uint8_t* xq = b + R.xq;
  uint8_t* xsf = b + R.xsf;
  float* xs = reinterpret_cast<float*>(b + R.xs);
  int32_t* counts = reinterpret_cast<int32_t*>(b + R.counts);
  int32_t* padded = reinterpret_cast<int32_t*>(b + R.padded);
  int32_t* r2s = reinterpret_cast<int32_t*>(b + R.r2s);
  void* fwd = b + R.fwd;
  // step marks: before the prologue (quantise + plan + permute), GEMM1, GEMM2, the combine,
  // and at the end; the forward's "before permute" and "before GEMM1" marks share one event
  void* fwd_events[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  if (num_step_events == 5) {
    if ((st = record_mark(step_events[0], s)) != MOE_OK) return st;
    fwd_events[0] = step_events[1];
    for (int i = 1; i < 5; ++i) fwd_events[i] = step_events[i];
  }
  const int id_mask = topk_ids_format == MOE_IDS_PACKED ? 0xFFFF : -1;
  const bool small = small_batch(M, top_k, d.H);
  if (small) {
    const WorkspaceLayout L = workspace_layout(d, M, top_k, do_finalize);
    uint8_t* fb = static_cast<uint8_t*>(fwd);
    const bool accum = do_finalize == MOE_OUTPUT_ACCUMULATE;
    const unsigned ctas = static_cast<unsigned>(M < kPrologueMaxCtas ? M : kPrologueMaxCtas);
    st = launch_pdl(small_prologue_kernel, dim3(ctas), dim3(kPrologueThreads), 0, s, x, static_cast<int>(M),
                    static_cast<int>(d.H), ld_x, act_scale_mode == MOE_SCALE_PER_TOKEN ? 1 : 0, topk_ids, id_mask,
                    static_cast<int>(top_k), static_cast<int>(local_expert_offset), static_cast<int>(d.El), xs,
                    counts, padded, r2s, token_to_row, dev_status, fb + L.aq, fb + L.asf,
                    reinterpret_cast<int32_t*>(fb + L.sched), reinterpret_cast<int32_t*>(fb + L.mtd),
                    static_cast<int>(counter_ints(L, L.mtd)), accum ? static_cast<const uint16_t*>(out) : nullptr,
                    accum ? reinterpret_cast<float*>(fb + L.g) : nullptr);
    if (st != MOE_OK) return st;
  } else {
    // the plan, then the quantiser storing straight into the plan rows (no permute launch)
    st = moe_plan(topk_ids, topk_ids_format, M, top_k, num_experts, local_expert_offset,
                  static_cast<int32_t>(d.El), counts, padded, r2s, token_to_row, b + R.plan_ws,
                  moe_plan_workspace_bytes(M, top_k, static_cast<int32_t>(d.El)), dev_status, stream);
    if (st != MOE_OK) return st;
    const WorkspaceLayout L = workspace_layout(d, M, top_k, do_finalize);
    uint8_t* fb = static_cast<uint8_t*>(fwd);
    const bool accum = do_finalize == MOE_OUTPUT_ACCUMULATE;
    // warps (tokens) per block: 8, fewer when a warp's H/16 x 9 staging bytes are large
    const int64_t stage_bytes = d.H / 16 * 9;
    int64_t wpb = (200 << 10) / stage_bytes;
    wpb = wpb > 8 ? 8 : wpb;
    MOE_CHECK(wpb >= 1, MOE_ERR_UNSUPPORTED_SHAPE);
    const size_t qs_smem = static_cast<size_t>(wpb * stage_bytes);
    if (qs_smem > (48 << 10))
      MOE_CUDA(cudaFuncSetAttribute(quantize_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(qs_smem)));
    const int64_t blocks = (static_cast<int64_t>(M) + wpb - 1) / wpb;
    const int64_t max_blocks = static_cast<int64_t>(num_sms()) * 16;
    st = launch_pdl(quantize_scatter_kernel, dim3(static_cast<unsigned>(blocks < max_blocks ? blocks : max_blocks)),
                    dim3(static_cast<unsigned>(wpb * 32)), qs_smem, s, x, static_cast<int>(M), static_cast<int>(d.H), ld_x,
                    act_scale_mode == MOE_SCALE_PER_TOKEN ? 1 : 0, static_cast<int>(top_k),
                    static_cast<const int32_t*>(token_to_row), xs, fb + L.aq, fb + L.asf,
                    reinterpret_cast<int32_t*>(fb + L.sched),
                    static_cast<int>(counter_ints(L, L.sched)), accum ? static_cast<const uint16_t*>(out) : nullptr,
                    accum ? reinterpret_cast<float*>(fb + L.g) : nullptr);
    if (st != MOE_OK) return st;
  }
  RoutingHint hint;
  hint.ids = topk_ids;
  hint.id_mask = id_mask;
  hint.off = local_expert_offset;
  hint.slots = M * top_k;
  return forward_chain(padded, r2s, token_to_row, M, top_k, xq, xsf, xs, w, prepared, topk_weights,
                       topk_weights_dtype, routed_scaling_factor, fc2_input_scale, do_finalize, out, gemm2_out, fwd,
                       dev_status, num_step_events == 5 ? fwd_events : nullptr, num_step_events, false, hint, topt, s);
}

extern "C" moe_status_t moe_routed_forward(const uint16_t* x, int32_t M, int64_t ld_x, int32_t act_scale_mode,
                                           const int32_t* topk_ids, int32_t topk_ids_format, int32_t top_k,
                                           int32_t num_experts, int32_t local_expert_offset, const void* topk_weights,
                                           int32_t topk_weights_dtype, float routed_scaling_factor,
                                           const moe_nvfp4_weights_t* w, const void* prepared, size_t prepared_bytes,
                                           float fc2_input_scale, int32_t do_finalize, uint16_t* out,
                                           uint16_t* gemm2_out, int32_t* token_to_row, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status, void* const* step_events,
                                           int32_t num_step_events, moe_stream_t stream) {
  return routed_forward(x, M, ld_x, act_scale_mode, topk_ids, topk_ids_format, top_k, num_experts,
                        local_expert_offset, topk_weights, topk_weights_dtype, routed_scaling_factor, w, prepared,
                        prepared_bytes, fc2_input_scale, do_finalize, out, gemm2_out, token_to_row, workspace,
                        workspace_bytes, dev_status, step_events, num_step_events, TestOptions(), stream);
}

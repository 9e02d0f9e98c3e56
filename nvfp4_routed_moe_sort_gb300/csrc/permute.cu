// S3 (permute), S7 (finalize) and the one-time weight layout preparation.
//
// Sources: FlashInfer flashinfer.fused_moe.CudnnGroupedGemmNvfp4Config (moe_permute: rows
// and scale rows permuted into expert order, scale rows rearranged into the GEMM's
// block-scale layout; moe_unpermute / finalize); FlashInfer
// flashinfer.fused_moe.FrostLowLatencyConfig (combine of ordered, separate FP32
// multiplications and additions; unrouted slots and their scores ignored); Megatron-Core
// core.inference.moe.flashinfer_nvfp4 (_pad_fc1: gate and up halves interleaved in row
// blocks so a GEMM tile sees both; prepare_routed_nvfp4_weights(out=...) refreshes in place).
#include <math.h>

#include "common.cuh"
#include "host_util.h"
#include "layout.h"

namespace moe {
namespace {

// One warp per plan row p < padded_offsets[El]: copy the token's packed row (16-byte
// vectors) and scatter its scale row into 128x4 tiles; scale columns past H/16 (K padding
// up to a multiple of 256) are written as zero. Padding rows are skipped: the GEMM rows
// they feed are never read. For an accumulated output, the same launch also copies the
// caller's BF16 out [M, H] into the FP32 accumulator that GEMM2 adds to.
__global__ void __launch_bounds__(256) permute_kernel(const int32_t* __restrict__ padded_offsets, int El,
                                                      const int32_t* __restrict__ row_to_slot, int top_k,
                                                      const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xsf,
                                                      int H, uint8_t* __restrict__ aq, uint8_t* __restrict__ asf,
                                                      int32_t* __restrict__ tile_counters,
                                                      int32_t* __restrict__ mt_done, int64_t n_mt,
                                                      const uint16_t* __restrict__ acc_init, float* __restrict__ acc,
                                                      int64_t acc_elems) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  // the GEMMs that follow claim their work units from these counters
  if (blockIdx.x == 0 && threadIdx.x < 2) tile_counters[threadIdx.x] = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_mt;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    mt_done[i] = 0;
  const int64_t P = padded_offsets[El];
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int row_bytes = H / 2;
  const int kcols = H / 16;
  const int kcols_p = static_cast<int>(roundup64(H, kTileK) / 16);
  for (int64_t p = warp0; p < P; p += nwarps) {
    const int s = row_to_slot[p];
    if (s < 0) continue;
    const int64_t t = s / top_k;
    const uint4* src = reinterpret_cast<const uint4*>(xq + t * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(aq + p * row_bytes);
    for (int v = lane; v < row_bytes / 16; v += 32) dst[v] = src[v];
    const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(xsf + t * kcols);
    for (int c4 = lane; c4 < kcols_p / 4; c4 += 32) {
      const uint32_t val = (c4 < kcols / 4) ? ssrc[c4] : 0u;
      *reinterpret_cast<uint32_t*>(asf + sf_tile_offset(p, 4 * c4, kcols_p)) = val;
    }
  }
  // accumulator = fp32(out), 8 values per thread and step
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = tid; i < acc_elems / 8; i += nthreads) {
    const uint4 v = reinterpret_cast<const uint4*>(acc_init)[i];
    float4* d = reinterpret_cast<float4*>(acc) + 2 * i;
    d[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xFFFF0000u));
    d[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u), __uint_as_float(v.w << 16),
                       __uint_as_float(v.w & 0xFFFF0000u));
  }
}

// out = bf16(acc), 8 values per thread
__global__ void __launch_bounds__(256) store_acc_kernel(const float* __restrict__ acc, int64_t elems,
                                                        uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < elems / 8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint32_t o[4];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k]))) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k + 1]))) << 16);
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// One warp per destination row of an expert matrix stack laid out for the GEMM:
// rows_p rows per expert (zero rows past the source rows), gated W1 with gate and up rows
// interleaved in 128-row blocks (destination rows [256n, 256n+128) = gate rows
// [128n, 128n+128), [256n+128, 256n+256) = up rows), scales in 128x4 tiles with K padded.
__global__ void __launch_bounds__(256) prepare_matrix_kernel(const uint8_t* __restrict__ src,
                                                             const uint8_t* __restrict__ src_sf, int E, int rows,
                                                             int rows_p, int K, int gated_inter,
                                                             uint8_t* __restrict__ dst, uint8_t* __restrict__ dst_sf) {
  const int lane = threadIdx.x & 31;
  const int64_t total = static_cast<int64_t>(E) * rows_p;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int row_bytes = K / 2;
  const int kcols = K / 16;
  const int kcols_p = static_cast<int>(roundup64(K, kTileK) / 16);
  const int64_t sf_expert_bytes = static_cast<int64_t>(rows_p) * kcols_p;
  for (int64_t r = warp0; r < total; r += nwarps) {
    const int e = static_cast<int>(r / rows_p);
    const int rr = static_cast<int>(r % rows_p);
    int sr;
    if (gated_inter > 0) {
      const int n = rr / 256, w = rr % 256;
      sr = (w < 128) ? n * 128 + w : gated_inter + n * 128 + (w - 128);
    } else {
      sr = rr;
    }
    const bool real = sr < rows;
    const int64_t srow = static_cast<int64_t>(e) * rows + sr;
    uint4* d = reinterpret_cast<uint4*>(dst + r * row_bytes);
    const uint4* sp = reinterpret_cast<const uint4*>(src + srow * row_bytes);
    for (int v = lane; v < row_bytes / 16; v += 32) d[v] = real ? sp[v] : make_uint4(0, 0, 0, 0);
    const uint32_t* ssp = reinterpret_cast<const uint32_t*>(src_sf + srow * kcols);
    uint8_t* dsf = dst_sf + e * sf_expert_bytes;
    for (int c4 = lane; c4 < kcols_p / 4; c4 += 32) {
      const uint32_t val = (real && c4 < kcols / 4) ? ssp[c4] : 0u;
      *reinterpret_cast<uint32_t*>(dsf + sf_tile_offset(rr, 4 * c4, kcols_p)) = val;
    }
  }
}

// out[t, :] = bf16(sum_j w[t,j] * row_j) with FP32 multiply and add kept separate and
// slots taken in ascending j. Each thread owns 8 consecutive columns of one token.
// BATCHED (few tokens, latency-bound): the loads of up to kMaxSlots slots are issued
// together before the ordered accumulation, so a token costs one or two memory round
// trips, not top_k. Otherwise (many tokens) the plain per-slot loop keeps more threads
// resident, which hides the latency better.
constexpr int kMaxSlots = 8;
constexpr int kBatchedFinalizeMaxTokens = 256;

template <bool BATCHED>
__global__ void __launch_bounds__(256) finalize_kernel(const uint16_t* __restrict__ rows,
                                                       const void* __restrict__ topk_weights, int weights_dtype,
                                                       float rsf, const int32_t* __restrict__ token_to_row, int M,
                                                       int top_k, int H, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int c8 = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= M || c8 * 8 >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  if constexpr (!BATCHED) {
    for (int j = 0; j < top_k; ++j) {
      const int r = token_to_row[static_cast<int64_t>(t) * top_k + j];
      if (r < 0) continue;
      const float w = route_weight(topk_weights, weights_dtype, static_cast<int64_t>(t) * top_k + j, rsf);
      const uint4 v = *reinterpret_cast<const uint4*>(rows + static_cast<int64_t>(r) * H + c8 * 8);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, __uint_as_float(u[i] << 16)));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, __uint_as_float(u[i] & 0xFFFF0000u)));
      }
    }
  }
  for (int j0 = 0; BATCHED && j0 < top_k; j0 += kMaxSlots) {
    int r[kMaxSlots];
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j)
      r[j] = (j0 + j < top_k) ? token_to_row[static_cast<int64_t>(t) * top_k + j0 + j] : -1;
    float w[kMaxSlots];
    uint4 v[kMaxSlots];
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      w[j] = 0.0f;
      v[j] = make_uint4(0, 0, 0, 0);
      if (r[j] >= 0) {
        w[j] = route_weight(topk_weights, weights_dtype, static_cast<int64_t>(t) * top_k + j0 + j, rsf);
        v[j] = *reinterpret_cast<const uint4*>(rows + static_cast<int64_t>(r[j]) * H + c8 * 8);
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      if (r[j] < 0) continue;
      const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w[j], __uint_as_float(u[i] << 16)));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w[j], __uint_as_float(u[i] & 0xFFFF0000u)));
      }
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
    o[i] = lo | (hi << 16);
  }
  *reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H + c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

int warp_grid(int64_t rows) {
  const int64_t blocks = (rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

moe_status_t launch_permute(const int32_t* padded_offsets, int El, const int32_t* row_to_slot, int top_k,
                            int64_t cap, const uint8_t* xq, const uint8_t* xsf, int H, uint8_t* aq, uint8_t* asf,
                            int32_t* tile_counters, int32_t* mt_done, int64_t n_mt, const uint16_t* acc_init,
                            float* acc, int64_t acc_elems, cudaStream_t s) {
  if (cap == 0) return MOE_OK;
  int grid = warp_grid(cap);
  const int64_t acc_blocks = (acc_elems / 8 + 255) / 256;
  const int64_t acc_cap = static_cast<int64_t>(num_sms()) * 8;
  if (acc_blocks > grid) grid = static_cast<int>(acc_blocks < acc_cap ? acc_blocks : acc_cap);
  return launch_pdl(permute_kernel, dim3(grid), dim3(256), 0, s, padded_offsets, El, row_to_slot, top_k, xq, xsf, H,
                    aq, asf, tile_counters, mt_done, n_mt, acc_init, acc, acc_elems);
}

moe_status_t launch_store_acc(const float* acc, int64_t elems, uint16_t* out, cudaStream_t s) {
  if (elems == 0) return MOE_OK;
  const int64_t blocks = (elems / 8 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  return launch_pdl(store_acc_kernel, dim3(static_cast<unsigned>(blocks < cap ? blocks : cap)), dim3(256), 0, s, acc,
                    elems, out);
}

moe_status_t launch_finalize(const uint16_t* rows, const void* topk_weights, int weights_dtype, float rsf,
                             const int32_t* token_to_row, int M, int top_k, int H, uint16_t* out, cudaStream_t s) {
  if (M == 0) return MOE_OK;
  const int threads = 256;
  const int bx = (H / 8 + threads - 1) / threads;
  if (M <= kBatchedFinalizeMaxTokens)
    return launch_pdl(finalize_kernel<true>, dim3(bx, M), dim3(threads), 0, s, rows, topk_weights, weights_dtype, rsf,
                      token_to_row, M, top_k, H, out);
  return launch_pdl(finalize_kernel<false>, dim3(bx, M), dim3(threads), 0, s, rows, topk_weights, weights_dtype, rsf,
                    token_to_row, M, top_k, H, out);
}

moe_status_t launch_prepare_matrix(const uint8_t* src, const uint8_t* src_sf, int E, int rows, int rows_p, int K,
                                   int gated_inter, uint8_t* dst, uint8_t* dst_sf, cudaStream_t s) {
  prepare_matrix_kernel<<<warp_grid(static_cast<int64_t>(E) * rows_p), 256, 0, s>>>(src, src_sf, E, rows, rows_p,
                                                                                    K, gated_inter, dst, dst_sf);
  return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_finalize(const uint16_t* gemm2_out, const void* topk_weights, int32_t topk_weights_dtype,
                                     float routed_scaling_factor, const int32_t* token_to_row, int32_t M,
                                     int32_t top_k, int32_t H, uint16_t* out, moe_stream_t stream) {
  MOE_CHECK(M >= 0 && top_k >= 1 && H > 0, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(topk_weights_dtype >= MOE_WEIGHTS_F32 && topk_weights_dtype <= MOE_WEIGHTS_PACKED,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(isfinite(routed_scaling_factor), MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(H % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(M < 65536, MOE_ERR_UNSUPPORTED_SHAPE);
  if (M == 0) return MOE_OK;
  MOE_CHECK(gemm2_out && topk_weights && token_to_row && out, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(gemm2_out) && aligned16(topk_weights) && aligned16(token_to_row) && aligned16(out),
            MOE_ERR_MISALIGNED);
  const size_t ob = static_cast<size_t>(M) * H * 2;
  const size_t wb = static_cast<size_t>(M) * top_k * (topk_weights_dtype == MOE_WEIGHTS_BF16 ? 2 : 4);
  MOE_CHECK(!overlaps(out, ob, topk_weights, wb) &&
                !overlaps(out, ob, token_to_row, static_cast<size_t>(M) * top_k * 4) &&
                !overlaps(out, ob, gemm2_out, 1),
            MOE_ERR_OVERLAP);
  return launch_finalize(gemm2_out, topk_weights, topk_weights_dtype, routed_scaling_factor,
                         token_to_row, M, top_k, H, out, as_stream(stream));
}

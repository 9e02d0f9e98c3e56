// S1: NVFP4 quantisation of BF16 rows (activations, per token or with global scale one)
// and of whole BF16 expert matrices (weights, one FP32 global scale per matrix).
//
// Sources: FlashInfer flashinfer.fused_moe.CudnnGroupedGemmNvfp4Config (Activations,
// prepare_activations: packed E2M1 [M, H/2], token-major E4M3 [M, H/16], global scale one);
// Megatron-Core core.inference.moe.flashinfer_nvfp4 (quantize_routed_nvfp4_input: one FP32
// scale per token; _global_encode_scale / _quantize_expert: one FP32 global scale per expert
// matrix; NVFP4_BLOCK_SIZE, FLOAT4_E2M1_MAX, FLOAT8_E4M3_MAX); vLLM flashinfer_utils
// (quantize_nvfp4_per_token_input: linear scale-factor layout).
//
// Few activation rows (up to 512) of up to 8192 values: one CTA per row with the row in
// registers (one global read, short latency chain). Otherwise one warp per row; the row is read once for its
// amax and once more, from L1/L2, for the blocks. Lane i handles 16-value blocks i, i+32,
// ...; each block is two 16-byte loads and one 8-byte store of codes, so a warp's loads and
// stores are contiguous.
#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

enum GScale : int { kGOne = 0, kGPerRow = 1, kGPerMatrix = 2 };

// rows [0, rows_total) of a [rows_total, ld] BF16 matrix -> data [rows_total, cols/2],
// sf [rows_total, cols/16]. Global encode scale per `gmode`; the decode scale goes to
// dec_out[row] (per row) or dec_out[row / rows_per_mat] (per matrix, written by the warp
// that owns the matrix's first row).
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows_total,
                                                            int cols, int64_t ld, int gmode,
                                                            const float* __restrict__ mat_amax,
                                                            int64_t rows_per_mat, uint8_t* __restrict__ data,
                                                            uint8_t* __restrict__ sf, float* __restrict__ dec_out) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int nblk = cols / kBlock;
  for (int64_t r = warp0; r < rows_total; r += nwarps) {
    const uint16_t* row = x + r * ld;
    float g = 1.0f, dec = 1.0f;
    if (gmode != kGOne) {
      float amax;
      if (gmode == kGPerRow) {
        amax = 0.0f;
        for (int b = lane; b < nblk; b += 32) {
          float v[16];
          load_block16(row + b * kBlock, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        amax = warp_max(amax);
      } else {
        amax = mat_amax[r / rows_per_mat];
      }
      if (amax > 0.0f) {
        g = __fdiv_rn(kGlobalNumerator, amax);
        dec = __fdiv_rn(amax, kGlobalNumerator);
      }
    }
    uint8_t* drow = data + r * (cols / 2);
    uint8_t* srow = sf + r * nblk;
    for (int b = lane; b < nblk; b += 32) {
      float v[16];
      load_block16(row + b * kBlock, v);
      uint32_t codes[2];
      const uint32_t q = quantize_block16(v, g, codes);
      *reinterpret_cast<uint2*>(drow + b * 8) = make_uint2(codes[0], codes[1]);
      srow[b] = static_cast<uint8_t>(q);
    }
    if (lane == 0) {
      if (gmode == kGPerRow || gmode == kGOne) {
        if (dec_out) dec_out[r] = dec;
      } else if (r % rows_per_mat == 0) {
        dec_out[r / rows_per_mat] = dec;
      }
    }
  }
}

// Rows of at most kRowCtaMaxCols values: one 128-thread CTA per row, each thread keeping up
// to four 16-value blocks in registers, so the row is read from global memory once; the
// per-token amax is a block reduction.
constexpr int kRowCtaThreads = 128;
constexpr int kRowCtaBlocks = 4;
constexpr int kRowCtaMaxCols = kRowCtaThreads * kRowCtaBlocks * kBlock;  // 8192
// with many rows the warp-per-row kernel keeps more loads in flight per SM and wins
constexpr int kRowCtaMaxRows = 512;

__global__ void __launch_bounds__(kRowCtaThreads) quantize_rows_cta_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int cols, int64_t ld, int per_row, uint8_t* __restrict__ data,
    uint8_t* __restrict__ sf, float* __restrict__ dec_out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kRowCtaThreads / 32];
  const int nblk = cols / kBlock;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint16_t* row = x + r * ld;
    float v[kRowCtaBlocks][16];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kRowCtaBlocks; ++j) {
      const int b = threadIdx.x + j * kRowCtaThreads;
      if (b < nblk) {
        load_block16(row + b * kBlock, v[j]);
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[j][i]));
      }
    }
    float g = 1.0f, dec = 1.0f;
    if (per_row) {
      amax = warp_max(amax);
      if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
      __syncthreads();
      amax = red[0];
#pragma unroll
      for (int w = 1; w < kRowCtaThreads / 32; ++w) amax = fmaxf(amax, red[w]);
      if (amax > 0.0f) {
        g = __fdiv_rn(kGlobalNumerator, amax);
        dec = __fdiv_rn(amax, kGlobalNumerator);
      }
    }
    uint8_t* drow = data + r * (cols / 2);
    uint8_t* srow = sf + r * nblk;
#pragma unroll
    for (int j = 0; j < kRowCtaBlocks; ++j) {
      const int b = threadIdx.x + j * kRowCtaThreads;
      if (b < nblk) {
        uint32_t codes[2];
        const uint32_t q = quantize_block16(v[j], g, codes);
        *reinterpret_cast<uint2*>(drow + b * 8) = make_uint2(codes[0], codes[1]);
        srow[b] = static_cast<uint8_t>(q);
      }
    }
    if (threadIdx.x == 0) dec_out[r] = dec;
    __syncthreads();  // red[] is reused by the next row
  }
}

// amax over each matrix (non-negative floats order like their bit patterns)
__global__ void __launch_bounds__(256) matrix_amax_kernel(const uint16_t* __restrict__ w, int64_t mat_elems,
                                                          float* __restrict__ amax) {
  const int mat = blockIdx.y;
  const uint16_t* base = w + static_cast<int64_t>(mat) * mat_elems;
  float m = 0.0f;
  const int64_t nvec = mat_elems / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = reinterpret_cast<const uint4*>(base)[i];
    const uint32_t ww[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m = fmaxf(m, fabsf(__uint_as_float(ww[k] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(ww[k] & 0xFFFF0000u)));
    }
  }
  m = warp_max(m);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(amax + mat), __float_as_uint(v));
  }
}

int rows_grid(int64_t rows) {
  const int64_t warps_needed = rows;
  const int64_t blocks = (warps_needed + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_quantize_input(const uint16_t* x, int32_t M, int32_t H, int64_t ld_x, int32_t mode,
                                           uint8_t* xq, uint8_t* xsf, float* xs, moe_stream_t stream) {
  MOE_CHECK(M >= 0 && H > 0 && ld_x >= H, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(mode == MOE_SCALE_GLOBAL_ONE || mode == MOE_SCALE_PER_TOKEN, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(H % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE);
  if (M == 0) return MOE_OK;
  MOE_CHECK(x && xq && xsf && xs, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(x) && aligned16(xq) && aligned16(xsf) && aligned16(xs) && ld_x % 8 == 0, MOE_ERR_MISALIGNED);
  const size_t xbytes = (static_cast<size_t>(M - 1) * ld_x + H) * 2;
  MOE_CHECK(!overlaps(x, xbytes, xq, static_cast<size_t>(M) * H / 2) &&
                !overlaps(x, xbytes, xsf, static_cast<size_t>(M) * H / 16) &&
                !overlaps(x, xbytes, xs, static_cast<size_t>(M) * 4),
            MOE_ERR_OVERLAP);
  if (H <= kRowCtaMaxCols && M <= kRowCtaMaxRows) {
    const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
    const unsigned grid = static_cast<unsigned>(M < cap ? M : cap);
    return launch_pdl(quantize_rows_cta_kernel, dim3(grid), dim3(kRowCtaThreads), 0, as_stream(stream), x,
                      static_cast<int64_t>(M), static_cast<int>(H), ld_x,
                      static_cast<int>(mode == MOE_SCALE_PER_TOKEN ? 1 : 0), xq, xsf, xs);
  }
  return launch_pdl(quantize_rows_kernel, dim3(rows_grid(M)), dim3(256), 0, as_stream(stream), x,
                    static_cast<int64_t>(M), static_cast<int>(H), ld_x,
                    static_cast<int>(mode == MOE_SCALE_PER_TOKEN ? kGPerRow : kGOne),
                    static_cast<const float*>(nullptr), static_cast<int64_t>(1), xq, xsf, xs);
}

extern "C" moe_status_t moe_quantize_weights(const uint16_t* w, int32_t num_mats, int32_t rows, int32_t cols,
                                             uint8_t* data, uint8_t* sf, float* alpha, float* amax_scratch,
                                             moe_stream_t stream) {
  MOE_CHECK(num_mats >= 0 && rows > 0 && cols > 0, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(cols % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE);
  if (num_mats == 0) return MOE_OK;
  MOE_CHECK(w && data && sf && alpha && amax_scratch, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(w) && aligned16(data) && aligned16(sf) && aligned16(alpha) && aligned16(amax_scratch),
            MOE_ERR_MISALIGNED);
  cudaStream_t s = as_stream(stream);
  const int64_t mat_elems = static_cast<int64_t>(rows) * cols;
  MOE_CUDA(cudaMemsetAsync(amax_scratch, 0, sizeof(float) * num_mats, s));
  int bx = static_cast<int>((mat_elems / 8 + 255) / 256);
  if (bx > 256) bx = 256;
  matrix_amax_kernel<<<dim3(bx, num_mats), 256, 0, s>>>(w, mat_elems, amax_scratch);
  MOE_CHECK(launch_status() == MOE_OK, MOE_ERR_CUDA);
  const int64_t rows_total = static_cast<int64_t>(num_mats) * rows;
  quantize_rows_kernel<<<rows_grid(rows_total), 256, 0, s>>>(w, rows_total, cols, cols, kGPerMatrix, amax_scratch,
                                                             rows, data, sf, alpha);
  return launch_status();
}

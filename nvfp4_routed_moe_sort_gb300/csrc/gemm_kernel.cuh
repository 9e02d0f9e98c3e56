// The grouped block-scaled NVFP4 GEMM kernel, a template over the epilogue mode and the
// activation (so every kernel carries only its own activation's code). Included by gemm.cu
// (launch set-up) and the gemm_inst_*.cu files (instantiations).
#pragma once

#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "host_util.h"
#include "layout.h"

namespace moe {
namespace gemm {

constexpr int kStages = 4;
constexpr int kABytes = kTileM * 128;           // 16 KB
constexpr int kBBytes = kTileN * 128;           // 32 KB
constexpr int kSfaBytes = 4 * 512;              // 2 KB: 4 scale tiles (one per K=64 step)
constexpr int kSfbBytes = 2 * 4 * 512;          // 4 KB: two 128-row halves
constexpr int kOffB = kABytes;
constexpr int kOffSfa = kABytes + kBBytes;
constexpr int kOffSfb = kOffSfa + kSfaBytes;
constexpr int kStageBytes = kOffSfb + kSfbBytes;  // 55296 = 54 KB
constexpr uint32_t kStageTx = kStageBytes;
constexpr int kTmemCols = 512;
constexpr int kSfCol0 = 256;
constexpr int kSfColsPerStage = 48;
// 16 warps in four warpgroups: warpgroup 0 = producer (warp 0), MMA issuer (warp 1) and two
// scale writers (warps 2, 3); warpgroups 1-2 = the eight epilogue warps (4-11); warpgroup 3
// = two scale writers (warps 12, 13) and two idle warps. A warp reaches only the TMEM lane
// quarter warp % 4, so the four writers (quarters 2, 3, 0, 1) cover all 128 lanes.
constexpr int kThreads = 512;
constexpr int kEpiThreads = 256;
constexpr int kEpiWarp0 = 4;
__host__ __device__ constexpr bool is_sf_writer(int warp) { return warp == 2 || warp == 3 || warp == 12 || warp == 13; }
constexpr int kSfWriters = 4;
// Register split (setmaxnreg): the epilogue warpgroups hold a tile's 128 accumulator columns
// per thread; the other two need few (72 keeps the producer's loop free of spills, which on
// its own slowed the launch by several percent). The launch gives 512 x 128 = 65536
// registers, and the split must not exceed that, or the raising warps would wait forever.
constexpr int kRegsAtLaunch = 128;
constexpr int kRegsEpi = 184;
constexpr int kRegsOther = 72;
static_assert(2 * 128 * kRegsEpi + 2 * 128 * kRegsOther <= kThreads * kRegsAtLaunch, "register split");
constexpr int kSmemExtra = 1024 /*align*/ + 256 /*barriers*/;
constexpr int kUnitRing = 4;      // work-unit ids handed from the producer to the other roles
// Tiles whose real rows all lie in the first kSparseRows rows (decode: a few tokens per
// expert) take the sparse epilogue: those rows' accumulators are staged in shared memory
// and every epilogue thread takes a share of the outputs.
constexpr int kSparseRows = 8;
constexpr int kSparseStageBytes = kSparseRows * kTileN * 4 + kSparseRows * 8;  // FP32 rows, slot + scalar
constexpr int kSparseMaxExperts = 384;  // above this the expert offsets leave no room for the stage
constexpr int kRingConsumers = 1 + kEpiThreads / 32 + kSfWriters;  // MMA thread, one lane per epilogue and writer warp

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
// barriers (full, empty, sf_full per stage; acc_full, acc_empty, final; the unit ring's two
// sets; stage_full, stage_empty), then the unit ring, the TMEM address and the abort flag
static_assert((3 * kStages + 3 + 2 * kUnitRing + 2) * 8 + kUnitRing * 4 + 8 <= 256, "barrier area");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

// One GEMM of the launch: operands, scales, per-expert scalars and output.
struct Phase {
  CUtensorMap tmap_a;     // 128-row activation boxes
  CUtensorMap tmap_a32;   // 32-row boxes, for tiles whose real rows all lie in the first 32
  CUtensorMap tmap_b;
  const uint8_t* b_raw;   // the weight rows behind tmap_b (K/2 bytes each), for the L2 prefetch
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* alpha;
  const float* alpha_gate;  // gate rows of a gated GEMM1
  void* out;
  uint8_t* out_sf;
  int32_t K, Kp, nkb, N, Np, n_tiles;
  int32_t out_v8;         // `out` is 32-byte aligned: BF16 rows go out in 32-byte stores
};

struct GemmParams {
  Phase ph[2];            // [1] only in the chained modes (GEMM2 after GEMM1 in one launch)
  const int32_t* padded_offsets;
  const int32_t* row_to_slot;
  const float* xs;
  int32_t* dev_status;
  int32_t* tile_counter;  // zeroed before the launch (by the permute kernel)
  int32_t* mt_done;       // chained modes: per 128-row tile, GEMM1 epilogue warps done (zeroed too)
  int32_t El, top_k, inter, gated, act;
  float g2;
  const void* route_w;  // kG2Reduce: route weights, their storage and the routed scaling factor
  int32_t route_w_dtype;
  float rsf;
  int32_t sparse;       // the sparse epilogue is enabled (shared memory holds its stage)
  uint64_t wait_ns;     // limit of every bounded wait (kWaitLimitNs unless a test build shortens it)
  int32_t withhold;     // test build only: GEMM1 tiles of row tile 0 never publish their completion
};

__host__ __device__ constexpr bool is_g2(int mode) { return mode == kG2Rows || mode == kG2Reduce; }
__host__ __device__ constexpr bool is_chain(int mode) { return mode == kChainRows || mode == kChainReduce; }
// epilogue of the first / second GEMM of a launch in `mode`
__host__ __device__ constexpr int first_epilogue(int mode) { return is_chain(mode) ? kG1Fused : mode; }
__host__ __device__ constexpr int second_epilogue(int mode) { return mode == kChainReduce ? kG2Reduce : kG2Rows; }

__device__ __forceinline__ void red_add_f32(float* out, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(out), "f"(v) : "memory");
}

// out[0..3] += v (FP32 additions performed at L2, in arrival order)
__device__ __forceinline__ void red_add_f32x4(float* out, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__host__ __device__ constexpr bool is_gated(int act) { return act == MOE_ACT_SWIGLU || act == MOE_ACT_GEGLU; }

__device__ __forceinline__ void decode_unit(int u, const int32_t* s_off, int El, int n_tiles, int& e, int& nt,
                                            int& mi) {
  int lo = 0, hi = El - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (n_tiles * (s_off[mid] >> 7) <= u) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int m_e = (s_off[e + 1] - s_off[e]) >> 7;
  const int local = u - n_tiles * (s_off[e] >> 7);
  nt = local / m_e;
  mi = local - nt * m_e;
}

// wait used only when shutting down after an abort: ignores the abort flag, short limit
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

__device__ __forceinline__ float silu_f32(float g) {
  return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
}

// GELU in its defining form x/2 * (1 + erf(x / sqrt(2)))
__device__ __forceinline__ float gelu_f32(float x) {
  return __fmul_rn(__fmul_rn(0.5f, x), __fadd_rn(1.0f, erff(__fmul_rn(x, 0.70710678118654752f))));
}

// Requantise 32 consecutive intermediate values (two 16-blocks) and store their 16 code
// bytes; returns the two scale bytes in bits [0,16).
__device__ __forceinline__ uint32_t requant32_store(const float* h, float g2, uint8_t* dst16) {
  uint32_t c0[2], c1[2];
  const uint32_t q0 = quantize_block16(h, g2, c0);
  const uint32_t q1 = quantize_block16(h + 16, g2, c1);
  *reinterpret_cast<uint4*>(dst16) = make_uint4(c0[0], c0[1], c1[0], c1[1]);
  return q0 | (q1 << 8);
}

// Pull this thread's 128 accumulator columns into registers, then hand the accumulator
// back to the MMA warp so the next tile's MMAs overlap this epilogue's arithmetic.
// Thread (lane quarter q, half h) owns TMEM lane 32q + lane and, for a gated GEMM1, gate
// columns [64h, 64h+64) plus the matching up columns [128+64h, ...); otherwise the columns
// [128h, 128h+128).
template <int MODE, int ACT>
__device__ __forceinline__ void load_acc(uint32_t tmem_row, int half, uint32_t* r, uint64_t* acc_empty) {
  if (!is_g2(MODE) && is_gated(ACT)) {
    tmem_ld32_issue(tmem_row + half * 64, r);
    tmem_ld32_issue(tmem_row + half * 64 + 32, r + 32);
    tmem_ld32_issue(tmem_row + 128 + half * 64, r + 64);
    tmem_ld32_issue(tmem_row + 128 + half * 64 + 32, r + 96);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32_issue(tmem_row + half * 128 + c * 32, r + 32 * c);
  }
  tmem_wait_ld<128>(r);
  tc_fence_before();
  mbar_arrive(acc_empty);
}

// 32 BF16 values (64 bytes) at dst: two 32-byte stores, each a whole L2 sector, when dst is
// 32-byte aligned (v8); else four 16-byte stores
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float* v, bool v8) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  if (v8) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * i), "r"(w[8 * i]),
                   "r"(w[8 * i + 1]), "r"(w[8 * i + 2]), "r"(w[8 * i + 3]), "r"(w[8 * i + 4]), "r"(w[8 * i + 5]),
                   "r"(w[8 * i + 6]), "r"(w[8 * i + 7])
                   : "memory");
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

template <int MODE, int ACT>
__device__ __forceinline__ void epilogue_compute(const GemmParams& p, const Phase& ph, uint32_t* r, int half,
                                                 int e, int nt,
                                                 int64_t prow, int slot, float xs_t) {
  constexpr bool kGated = is_gated(ACT);
  const bool real = slot >= 0;
  if constexpr (MODE == kG2Rows) {
    const float d2 = __fmul_rn(ph.alpha[e], __fdiv_rn(1.0f, p.g2));
    const int col0 = nt * kTileN + half * 128;
    if (!real || col0 >= ph.N) return;
    uint16_t* orow = static_cast<uint16_t*>(ph.out) + prow * ph.N + col0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(__uint_as_float(r[32 * c + i]), d2);
      store_bf16x32(orow + 32 * c, v, ph.out_v8);
    }
  } else if constexpr (MODE == kG2Reduce) {
    // acc[t, :] += (y2 * w') for this row's token t, w' = fp32(w * rsf)
    const float d2 = __fmul_rn(ph.alpha[e], __fdiv_rn(1.0f, p.g2));
    const int col0 = nt * kTileN + half * 128;
    if (!real || col0 >= ph.N) return;
    const float w = route_weight(p.route_w, p.route_w_dtype, slot, p.rsf);
    float* orow = static_cast<float*>(ph.out) + static_cast<int64_t>(slot / p.top_k) * ph.N + col0;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __fmul_rn(__fmul_rn(__uint_as_float(r[4 * c + i]), d2), w);
      red_add_f32x4(orow + 4 * c, v[0], v[1], v[2], v[3]);
    }
  } else {
    if (!real) return;
    const float a1 = ph.alpha[e];
    const float a1g = kGated ? ph.alpha_gate[e] : a1;  // gate rows' scalar
    const int I = p.inter;
    const int ip16 = static_cast<int>(roundup64(I, kTileK) / 16);  // scale columns of the intermediate
    // intermediate columns [i0, i0 + nout) come from this thread's registers
    const int i0 = kGated ? nt * 128 + half * 64 : nt * kTileN + half * 128;
    const int nout = kGated ? 64 : 128;
    if (i0 >= I) return;
    if constexpr (MODE == kG1Preact) {
      const int ld = kGated ? 2 * I : I;
      float* o = static_cast<float*>(ph.out) + prow * ld;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        const float y = __fmul_rn(__fmul_rn(__uint_as_float(r[i]), xs_t), i < nout ? a1g : a1);
        if (i < nout) o[i0 + i] = y;                    // gate (or all) columns
        else if (kGated) o[I + i0 + i - 64] = y;        // up columns
      }
      return;
    }
    // activation, 32 intermediate values at a time
    uint32_t sfw = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c * 32 >= nout) break;
      float h[32];
      // the activation is a compile-time constant: each kernel carries only its own code
#define MOE_Y(idx) __fmul_rn(__fmul_rn(__uint_as_float(r[idx]), xs_t), a1)
#define MOE_YG(idx) __fmul_rn(__fmul_rn(__uint_as_float(r[idx]), xs_t), a1g)
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if constexpr (ACT == MOE_ACT_SWIGLU) {
          h[i] = bf16_round_f32(__fmul_rn(silu_f32(MOE_YG(32 * c + i)), MOE_Y(64 + 32 * c + i)));
        } else if constexpr (ACT == MOE_ACT_GEGLU) {
          h[i] = bf16_round_f32(__fmul_rn(gelu_f32(MOE_YG(32 * c + i)), MOE_Y(64 + 32 * c + i)));
        } else if constexpr (ACT == MOE_ACT_RELU2) {
          const float t = fmaxf(MOE_Y(32 * c + i), 0.0f);
          h[i] = bf16_round_f32(__fmul_rn(t, t));
        } else if constexpr (ACT == MOE_ACT_GELU) {
          h[i] = bf16_round_f32(gelu_f32(MOE_Y(32 * c + i)));
        } else if constexpr (ACT == MOE_ACT_SILU) {
          h[i] = bf16_round_f32(silu_f32(MOE_Y(32 * c + i)));
        } else if constexpr (ACT == MOE_ACT_RELU) {
          h[i] = bf16_round_f32(fmaxf(MOE_Y(32 * c + i), 0.0f));
        } else {
          h[i] = bf16_round_f32(MOE_Y(32 * c + i));
        }
      }
#undef MOE_Y
#undef MOE_YG
      const int ic = i0 + 32 * c;
      if constexpr (MODE == kG1Act) {
        store_bf16x32(static_cast<uint16_t*>(ph.out) + prow * I + ic, h, ph.out_v8);
      } else {
        uint8_t* dst = static_cast<uint8_t*>(ph.out) + prow * (I / 2) + ic / 2;
        const uint32_t q2 = requant32_store(h, p.g2, dst);
        // two 32-value chunks make one 4-scale group of the 128x4 tile layout
        if (c & 1) {
          *reinterpret_cast<uint32_t*>(ph.out_sf + sf_tile_offset(prow, (ic >> 4) - 2, ip16)) = sfw | (q2 << 16);
        } else {
          sfw = q2;
        }
      }
    }
    if constexpr (MODE == kG1Fused) {
      // zero the scale columns of the K padding once per row (last column tile, first half)
      if (nt == ph.n_tiles - 1 && half == 0) {
        for (int c4 = I / 64; c4 < ip16 / 4; ++c4)
          *reinterpret_cast<uint32_t*>(ph.out_sf + sf_tile_offset(prow, 4 * c4, ip16)) = 0u;
      }
    }
  }
}

// The activation of GEMM1 on one output: gated kinds take the gate and up pre-activations.
template <int ACT>
__device__ __forceinline__ float activation_f32(float yg, float yu) {
  if constexpr (ACT == MOE_ACT_SWIGLU) return __fmul_rn(silu_f32(yg), yu);
  else if constexpr (ACT == MOE_ACT_GEGLU) return __fmul_rn(gelu_f32(yg), yu);
  else if constexpr (ACT == MOE_ACT_RELU2) {
    const float t = fmaxf(yg, 0.0f);
    return __fmul_rn(t, t);
  } else if constexpr (ACT == MOE_ACT_GELU) return gelu_f32(yg);
  else if constexpr (ACT == MOE_ACT_SILU) return silu_f32(yg);
  else if constexpr (ACT == MOE_ACT_RELU) return fmaxf(yg, 0.0f);
  else return yg;
}

// The arithmetic of the sparse epilogue on the staged rows (nrows leading real rows). With
// `dry` it runs one pass on whatever the stage holds and stores nothing: a kernel runs it
// once before its first tile arrives, so the code and the expert scalars are cached by then.
template <int MODE, int ACT>
__device__ __noinline__ void sparse_compute(const GemmParams& p, const Phase& ph, int etid, int e, int nt,
                                            int64_t row0, int nrows, const float* s_stage, const int32_t* s_slot,
                                            const float* s_scal, bool dry) {
  constexpr bool kGated = is_gated(ACT);
  const float a1 = ph.alpha[e];
  const float a1g = (!is_g2(MODE) && kGated) ? ph.alpha_gate[e] : a1;
  if constexpr (is_g2(MODE)) {
    const float d2 = __fmul_rn(a1, __fdiv_rn(1.0f, p.g2));
    const int n_out = nrows * kTileN;
    for (int o = etid; o < n_out; o += kEpiThreads) {
      const int row = o >> 8, j = o & (kTileN - 1);
      const int col = nt * kTileN + j;
      if (col >= ph.N) continue;
      const float y = __fmul_rn(s_stage[row * kTileN + j], d2);
      if constexpr (MODE == kG2Rows) {
        const uint16_t v = __bfloat16_as_ushort(__float2bfloat16_rn(y));
        if (!dry) static_cast<uint16_t*>(ph.out)[(row0 + row) * ph.N + col] = v;
      } else {
        const int t = s_slot[row] / p.top_k;
        const float v = __fmul_rn(y, s_scal[row]);
        if (!dry) red_add_f32(static_cast<float*>(ph.out) + static_cast<int64_t>(t) * ph.N + col, v);
      }
    }
  } else {
    const int I = p.inter;
    const int ip16 = static_cast<int>(roundup64(I, kTileK) / 16);
    constexpr int kOut = kGated ? 128 : kTileN;  // intermediate columns per row of the tile
    const int n_out = nrows * kOut;
    uint8_t* out = static_cast<uint8_t*>(ph.out);
    // every lane runs every pass (the block max is a warp shuffle); 16-lane groups are
    // wholly valid or wholly not
    for (int o0 = 0; o0 < n_out; o0 += kEpiThreads) {
      const int o = o0 + etid;
      const int row = (o / kOut) & (kSparseRows - 1);
      const int j = o % kOut;
      const int ic = kGated ? nt * 128 + j : nt * kTileN + j;
      const bool valid = o < n_out && ic < I;
      float h = 0.0f;
      if (valid) {
        const float xs_t = s_scal[row];
        const float* st = s_stage + row * kTileN;
        const float yg = __fmul_rn(__fmul_rn(st[j], xs_t), kGated ? a1g : a1);
        const float yu = kGated ? __fmul_rn(__fmul_rn(st[128 + j], xs_t), a1) : 0.0f;
        h = bf16_round_f32(activation_f32<ACT>(yg, yu));
      }
      float amax = fmaxf(0.0f, fabsf(h));
#pragma unroll
      for (int m = 8; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      const float sc = __fmul_rn(__fdiv_rn(amax, 6.0f), p.g2);
      const uint32_t qs = f32_to_e4m3(sc);
      const float qf = e4m3_to_f32(qs);
      const float inv = (qf == 0.0f) ? 0.0f : __fdiv_rn(p.g2, qf);
      const float hn = __shfl_down_sync(0xffffffffu, h, 1);
      if (valid && !dry) {
        const int64_t prow = row0 + row;
        if ((j & 1) == 0) out[prow * (I / 2) + ic / 2] = static_cast<uint8_t>(f32x2_to_e2m1(__fmul_rn(h, inv), __fmul_rn(hn, inv)));
        if ((j & 15) == 0) ph.out_sf[sf_tile_offset(prow, ic >> 4, ip16)] = static_cast<uint8_t>(qs);
      }
    }
    // zero the scale columns of the K padding once per real row (last column tile)
    if (!dry && nt == ph.n_tiles - 1 && etid < nrows) {
      for (int c4 = I / 64; c4 < ip16 / 4; ++c4)
        *reinterpret_cast<uint32_t*>(ph.out_sf + sf_tile_offset(row0 + etid, 4 * c4, ip16)) = 0u;
    }
  }
}

// Sparse epilogue of one work unit (all its real rows among the first kSparseRows rows).
// The two warps that own TMEM lanes 0-31 copy the real rows' 256 accumulator columns into
// the shared stage and release the accumulator; then all 256 epilogue threads share the
// outputs: thread o of a pass handles output o (consecutive threads = consecutive columns
// of a row), so a 16-value requant block is 16 lanes of one warp (block max by shuffles).
// The arithmetic per value is the dense epilogue's. Returns false after an aborted wait.
template <int MODE, int ACT>
__device__ __noinline__ bool sparse_epilogue(const GemmParams& p, const Phase& ph, uint32_t tmem_row, int q, int half,
                                             int lane,
                                                int etid, int e, int nt, int64_t row0, int slot, float scal,
                                                float* s_stage, int32_t* s_slot, float* s_scal, uint64_t* acc_empty,
                                                uint64_t* stage_full, uint64_t* stage_empty, uint32_t& sphase,
                                                volatile int* abort_flag) {
  if (q == 0) {
    bool ok = mbar_wait(stage_empty, sphase ^ 1, abort_flag, p.dev_status, p.wait_ns);
    if (!__all_sync(0xffffffffu, ok)) return false;
    // 32 columns at a time (few registers: this path runs inside the dense epilogue's loop)
    float4* dst = reinterpret_cast<float4*>(s_stage + (lane & (kSparseRows - 1)) * kTileN + half * 128);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t acc[32];
      tmem_ld32_issue(tmem_row + half * 128 + c * 32, acc);
      tmem_wait_ld<32>(acc);
      if (lane < kSparseRows) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          dst[c * 8 + v] = make_float4(__uint_as_float(acc[4 * v]), __uint_as_float(acc[4 * v + 1]),
                                       __uint_as_float(acc[4 * v + 2]), __uint_as_float(acc[4 * v + 3]));
      }
    }
    tc_fence_before();
    mbar_arrive(acc_empty);
    if (lane < kSparseRows) {
      if (half == 0) {
        s_slot[lane] = slot;
        s_scal[lane] = scal;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(stage_full);
  } else {
    tc_fence_before();
    mbar_arrive(acc_empty);
  }
  bool ok = mbar_wait(stage_full, sphase, abort_flag, p.dev_status, p.wait_ns);
  if (!__all_sync(0xffffffffu, ok)) return false;
  sphase ^= 1;
  int nrows = 0;  // real rows lead the tile
#pragma unroll
  for (int i = 0; i < kSparseRows; ++i) nrows += s_slot[i] >= 0 ? 1 : 0;
  sparse_compute<MODE, ACT>(p, ph, etid, e, nt, row0, nrows, s_stage, s_slot, s_scal, false);
  __syncwarp();
  if (lane == 0) mbar_arrive(stage_empty);
  return true;
}

// Bounded wait until *counter >= target (acquire): the GEMM2 half of a chained launch waits
// here for the GEMM1 tiles it reads. Gives up like mbar_wait.
__device__ __forceinline__ bool wait_counter(const int32_t* counter, int target, volatile int* abort_flag,
                                             int32_t* dev_status, uint64_t limit_ns) {
  uint64_t t0 = 0;
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    if (*abort_flag) return false;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > limit_ns) {
      *abort_flag = 1;
      if (dev_status) atomicOr(dev_status, MOE_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
}

// *counter += v with release semantics at GPU scope: the warp's earlier writes (ordered before
// this lane's by __syncwarp) are visible to whoever acquires the new count
__device__ __forceinline__ void red_release_add(int32_t* counter, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(counter), "r"(v) : "memory");
}

// orders this thread's generic-proxy global accesses with its async-proxy (TMA) ones
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// L2 prefetch of a contiguous range (16-byte aligned, multiple of 16 bytes) in 64 KB requests
__device__ __forceinline__ void prefetch_l2(const uint8_t* ptr, int64_t bytes) {
  for (int64_t o = 0; o < bytes; o += 65536) {
    const int64_t n = bytes - o < 65536 ? bytes - o : 65536;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr + o), "r"(static_cast<uint32_t>(n))
                 : "memory");
  }
}

// Epilogue of one work unit `uu` of GEMM `ph` (epilogue kind EK): wait for the accumulator,
// then the sparse or the dense epilogue. Returns false after an aborted wait; row0 = the
// unit's first plan row.
template <int EK, int ACT>
__device__ __forceinline__ bool epilogue_unit(const GemmParams& p, const Phase& ph, int uu, const int32_t* s_off,
                                              uint32_t tmem_row, int q, int half, int lane, int r, int etid,
                                              uint32_t& acc_phase, uint32_t& sphase, float* s_stage, int32_t* s_slot,
                                              float* s_scal, uint64_t* acc_full, uint64_t* acc_empty,
                                              uint64_t* stage_full, uint64_t* stage_empty, volatile int* abort_flag,
                                              int64_t& row0) {
  int e, nt, mi;
  decode_unit(uu, s_off, p.El, ph.n_tiles, e, nt, mi);
  row0 = s_off[e] + mi * kTileM;
  const int64_t prow = row0 + r;
  const int slot = p.row_to_slot[prow];
  const float xs_t = (!is_g2(EK) && slot >= 0) ? p.xs[slot / p.top_k] : 0.0f;
  const bool sparse = (EK == kG1Fused || is_g2(EK)) && p.sparse && p.row_to_slot[row0 + kSparseRows] < 0;
  float scal = xs_t;
  if constexpr (EK == kG2Reduce) scal = slot >= 0 ? route_weight(p.route_w, p.route_w_dtype, slot, p.rsf) : 0.0f;
  bool ok = mbar_wait(acc_full, acc_phase, abort_flag, p.dev_status, p.wait_ns);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  tc_fence_after();
  acc_phase ^= 1;
  if (sparse)
    return sparse_epilogue<EK, ACT>(p, ph, tmem_row, q, half, lane, etid, e, nt, row0, slot, scal, s_stage, s_slot,
                                    s_scal, acc_empty, stage_full, stage_empty, sphase, abort_flag);
  uint32_t acc[128];
  load_acc<EK, ACT>(tmem_row, half, acc, acc_empty);
  if (__any_sync(0xffffffffu, slot >= 0)) epilogue_compute<EK, ACT>(p, ph, acc, half, e, nt, prow, slot, xs_t);
  return true;
}

template <int MODE, int ACT>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr bool kChain = is_chain(MODE);
  constexpr int kEpi0 = first_epilogue(MODE);
  constexpr int kEpi1 = second_epilogue(MODE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* final_bar = acc_empty + 1;
  uint64_t* unit_full = final_bar + 1;
  uint64_t* unit_empty = unit_full + kUnitRing;
  uint64_t* stage_full = unit_empty + kUnitRing;
  uint64_t* stage_empty = stage_full + 1;
  uint64_t* sf_full = stage_empty + 1;  // per stage: its scales are in TMEM (one arrival per writer warp)
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(sf_full + kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + kStages) + kUnitRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + 256);
  // sparse-epilogue stage: [kSparseRows][kTileN] FP32, then per-row slot and scalar
  float* s_stage = reinterpret_cast<float*>(smem + kStages * kStageBytes + 256 + roundup64((p.El + 1) * 4, 16));
  int32_t* s_slot = reinterpret_cast<int32_t*>(s_stage + kSparseRows * kTileN);
  float* s_scal = reinterpret_cast<float*>(s_slot + kSparseRows);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool epi_warp = warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiThreads / 32;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], kSfWriters);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiThreads);
    mbar_init(final_bar, 1);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&unit_full[i], 1);
      mbar_init(&unit_empty[i], kRingConsumers);
    }
    mbar_init(stage_full, 2);                  // the two warps holding TMEM lanes 0-31
    mbar_init(stage_empty, kEpiThreads / 32);  // one arrival per epilogue warp
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < (kChain ? 2 : 1); ++i) {
      prefetch_tensormap(&p.ph[i].tmap_a);
      prefetch_tensormap(&p.ph[i].tmap_a32);
      prefetch_tensormap(&p.ph[i].tmap_b);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();  // the plan, activations and tile counter come from earlier kernels
  // the producer's first claim goes out now (its round trip overlaps the plan load); each
  // later claim is issued one unit early, while the current unit's loads go out
  int next_claim = 0;
  if (threadIdx.x == 0) next_claim = atomicAdd(p.tile_counter, 1);
  for (int i = threadIdx.x; i <= p.El; i += blockDim.x) s_off[i] = p.padded_offsets[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // units [0, units0) belong to the first GEMM, [units0, total_units) to the second (chained)
  const int mtiles = s_off[p.El] >> 7;
  const int units0 = mtiles * p.ph[0].n_tiles;
  const int total_units = units0 + (kChain ? mtiles * p.ph[1].n_tiles : 0);
  // the producer claims work units and hands their ids to the MMA and epilogue warps
  auto take_unit = [&](uint32_t& rslot, uint32_t& rphase, bool one_lane) -> int {
    bool got = mbar_wait(&unit_full[rslot], rphase, abort_flag, p.dev_status, p.wait_ns);
    if (!one_lane) got = __all_sync(0xffffffffu, got);
    if (!got) return -2;
    const int u = unit_ring[rslot];
    if (!one_lane) __syncwarp();
    if (one_lane || lane == 0) mbar_arrive(&unit_empty[rslot]);
    if (++rslot == kUnitRing) { rslot = 0; rphase ^= 1; }
    return u;
  };

  if (!epi_warp) {
    // warpgroups 0 and 3 give up registers first; the epilogue's raise draws on them
    setmaxnreg_dec<kRegsOther>();
    if (warp == 0) {
      if (lane == 0) {
        uint32_t stage = 0, phase = 0;
        uint32_t issued_mask = 0, issued_phase = 0;
        uint32_t rslot = 0, rphase = 0;
        bool ok = true;
        while (ok) {
          // claim the next unit (in order, from the global counter) and publish its id
          if (!mbar_wait(&unit_empty[rslot], rphase ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
          // claims increase per CTA, so a GEMM2 tile never waits behind a GEMM1 tile that its
          // own CTA has claimed but not started
          int u = next_claim;
          next_claim = atomicAdd(p.tile_counter, 1);
          if (u >= total_units) u = -1;
          unit_ring[rslot] = u;
          mbar_arrive(&unit_full[rslot]);
          if (++rslot == kUnitRing) { rslot = 0; rphase ^= 1; }
          if (u < 0) break;
          const bool second = kChain && u >= units0;
          const Phase& ph = p.ph[second ? 1 : 0];
          int e, nt, mi;
          decode_unit(second ? u - units0 : u, s_off, p.El, ph.n_tiles, e, nt, mi);
          const int row0 = s_off[e] + mi * kTileM;
          const int brow0 = e * ph.Np + nt * kTileN;
          const int64_t kt = ph.Kp >> 6;  // 512-byte scale tiles per 128 rows
          const uint8_t* sfa = ph.sfa + static_cast<int64_t>(row0 >> 7) * kt * 512;
          const uint8_t* sfb0 = ph.sfb + (static_cast<int64_t>(e) * (ph.Np >> 7) + nt * 2) * kt * 512;
          const uint8_t* sfb1 = sfb0 + kt * 512;
          if (second) {
            // wait until every GEMM1 tile of these rows has been written; if they are not yet,
            // the weight tile and its scales (which do not depend on GEMM1) start towards L2
            const int32_t* done = p.mt_done + (row0 >> 7);
            const int target = (kEpiThreads / 32) * p.ph[0].n_tiles;
            int seen;
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(seen) : "l"(done) : "memory");
            if (seen < target) {
              prefetch_l2(ph.b_raw + static_cast<int64_t>(brow0) * (ph.K / 2),
                          static_cast<int64_t>(kTileN) * (ph.K / 2));
              prefetch_l2(sfb0, 2 * kt * 512);
              if (!wait_counter(done, target, abort_flag, p.dev_status, p.wait_ns)) {
                ok = false;
                break;
              }
            }
            fence_proxy_async_global();  // the TMA reads below follow the observed generic writes
          }
          // a tile whose row 32 is padding has all its real rows in the first 32 (padding rows
          // end a segment): load only those; the MMA rows fed by stale shared memory are
          // padding rows, whose results are never stored
          const bool short_tile = p.row_to_slot[row0 + 32] < 0;
          const uint32_t tx = short_tile ? kStageTx - (kABytes - 32 * 128) : kStageTx;
          for (int kb = 0; kb < ph.nkb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
            uint8_t* st = smem + stage * kStageBytes;
            mbar_arrive_expect_tx(&full[stage], tx);
            tma_load_2d(st, short_tile ? &ph.tmap_a32 : &ph.tmap_a, kb * 128, row0, &full[stage]);
            tma_load_2d(st + kOffB, &ph.tmap_b, kb * 128, brow0, &full[stage]);
            bulk_load(st + kOffSfa, sfa + kb * 2048, 2048, &full[stage]);
            bulk_load(st + kOffSfb, sfb0 + kb * 2048, 2048, &full[stage]);
            bulk_load(st + kOffSfb + 2048, sfb1 + kb * 2048, 2048, &full[stage]);
            issued_mask |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
        }
        // copies may still be landing in shared memory (after an abort, or when another role
        // gave up before consuming them): let every issued stage land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (issued_mask & (1u << s)) mbar_drain(&full[s], (issued_phase >> s) & 1);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_mxf4nvf4(kTileM, kTileN);
        uint32_t stage = 0, phase = 0, acc_phase = 0;
        uint32_t rslot = 0, rphase = 0;
        bool ok = true;
        while (ok) {
          const int u = take_unit(rslot, rphase, true);
          if (u < 0) break;
          if (!mbar_wait(acc_empty, acc_phase ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const int nkb = p.ph[kChain && u >= units0 ? 1 : 0].nkb;
          for (int kb = 0; kb < nkb; ++kb) {
            // the stage's operands have landed and the writer warps have put its scales in TMEM
            if (!mbar_wait(&sf_full[stage], phase, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + stage * kStageBytes);
            const uint32_t sft = tmem + kSfCol0 + stage * kSfColsPerStage;
            // one M=128, N=256, K=64 MMA per K step: the 256-row B tile is one operand (8-row
            // groups 1024 bytes apart, so its second half follows the first)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_mxf4nvf4(tmem, sdesc_kmajor_sw128(st + kk * 32), sdesc_kmajor_sw128(st + kOffB + kk * 32), idesc,
                           sft + kk * 4, sft + 16 + kk * 8, (kb | kk) != 0);
            tc_commit(&empty[stage]);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          tc_commit(acc_full);
          acc_phase ^= 1;
        }
        // every MMA issued by this thread has finished before TMEM is released
        tc_commit(final_bar);
        mbar_drain(final_bar, 0);
      }
    } else if (is_sf_writer(warp)) {
      // Scale writers: per stage, once its copies have landed, each writer warp stores the
      // stage's scale atoms into its own TMEM lane quarter (tcgen05.st), the layout the
      // MMAs read: A's 4 atoms (one per K=64 step) in columns [0, 16); B's in [16, 48), the
      // two 128-row halves of a K step side by side (8 columns per step). Line l of a 512-byte
      // atom (16 bytes: the scales of rows l, l+32, l+64, l+96) goes to lane l of every
      // quarter, as a replicating copy of the atom would put it. This keeps the MMA thread's
      // instruction stream to the MMAs alone. A stage's scale columns are free once its
      // operands have landed: the producer reloads a stage only after the MMAs that read it
      // (and its scale columns) have completed.
      const uint32_t sf_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kSfCol0;
      uint32_t stage = 0, phase = 0;
      uint32_t rslot = 0, rphase = 0;
      bool ok = true;
      while (ok) {
        const int u = take_unit(rslot, rphase, false);
        if (u < 0) break;
        const int nkb = p.ph[kChain && u >= units0 ? 1 : 0].nkb;
        for (int kb = 0; kb < nkb; ++kb) {
          const bool got = mbar_wait(&full[stage], phase, abort_flag, p.dev_status, p.wait_ns);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          // 16 columns per store (A's four atoms; then B's K steps 0-1 and 2-3)
          const uint4* atoms = reinterpret_cast<const uint4*>(smem + stage * kStageBytes + kOffSfa);
          const uint32_t sft = sf_lane + stage * kSfColsPerStage;
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            uint32_t v[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              // part 0: A atom i; parts 1-2: B atom (K step 2(part-1) + i/2, half i%2)
              const int atom = part == 0 ? i : 4 + (i & 1) * 4 + (part - 1) * 2 + (i >> 1);
              const uint4 w = atoms[atom * 32 + lane];
              v[4 * i] = w.x; v[4 * i + 1] = w.y; v[4 * i + 2] = w.z; v[4 * i + 3] = w.w;
            }
            tmem_st16(sft + 16 * part, v);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sf_full[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else {
    setmaxnreg_inc<kRegsEpi>();
    if (p.sparse) {
      // before the first accumulator is ready: one dry pass of the sparse epilogue (expert 0),
      // which brings its code and the scalar tables into the caches. (Called here, under the
      // epilogue's register budget: a call before the role split made the compiler keep values
      // of the epilogue loop on the stack.)
      if constexpr (kEpi0 == kG1Fused || is_g2(kEpi0))
        sparse_compute<kEpi0, ACT>(p, p.ph[0], threadIdx.x - kEpiWarp0 * 32, 0, 0, 0, 1, s_stage, s_slot, s_scal,
                                   true);
      if constexpr (kChain)
        sparse_compute<kEpi1, MOE_ACT_IDENTITY>(p, p.ph[1], threadIdx.x - kEpiWarp0 * 32, 0, 0, 0, 1, s_stage,
                                                s_slot, s_scal, true);
    }
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = (warp - kEpiWarp0) >> 2;  // column half of the tile
    const int r = q * 32 + lane;            // row inside the 128-row tile
    const uint32_t tmem_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t acc_phase = 0, sphase = 0;
    uint32_t rslot = 0, rphase = 0;
    const int etid = threadIdx.x - kEpiWarp0 * 32;  // 0..255 over the epilogue warps
    while (true) {
      const int u = take_unit(rslot, rphase, false);
      if (u < 0) break;
      int64_t row0 = 0;
      bool first = true;
      if constexpr (kChain) first = u < units0;
      if (first) {
        if (!epilogue_unit<kEpi0, ACT>(p, p.ph[0], u, s_off, tmem_row, q, half, lane, r, etid, acc_phase, sphase,
                                       s_stage, s_slot, s_scal, acc_full, acc_empty, stage_full, stage_empty,
                                       abort_flag, row0))
          break;
        if (kChain) {
          // this warp's share of a GEMM1 tile is written: publish it to the GEMM2 tiles
          __syncwarp();
          if (lane == 0 && !(p.withhold && row0 < kTileM)) red_release_add(p.mt_done + (row0 >> 7), 1);
        }
      } else if constexpr (kChain) {
        if (!epilogue_unit<kEpi1, MOE_ACT_IDENTITY>(p, p.ph[1], u - units0, s_off, tmem_row, q, half, lane, r, etid,
                                                    acc_phase, sphase, s_stage, s_slot, s_scal, acc_full, acc_empty,
                                                    stage_full, stage_empty, abort_flag, row0))
          break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE, int ACT>
moe_status_t launch_kernel(const GemmParams& prm, int64_t units_max, size_t smem, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<MODE, ACT>;
  // the register split is drawn from what the launch provides: refuse a build that gives less
  cudaFuncAttributes fa;
  MOE_CUDA(cudaFuncGetAttributes(&fa, kern));
  if (fa.numRegs < kRegsAtLaunch) return MOE_ERR_CUDA;
  MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
  // persistent: one CTA per SM, at most one per work unit
  const int grid = static_cast<int>(units_max < num_sms() ? units_max : num_sms());
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, prm);
}

// launch set-up shared by the chained launcher (gemm.cu) and the test build's standalone GEMM1
bool fill_phase(Phase& ph, const GemmLaunch& g);
void fill_common(GemmParams& prm, const GemmLaunch& g);
size_t smem_bytes(int64_t El, bool sparse);

// instantiated in the gemm_inst_chain_*.cu files
moe_status_t launch_chain_gated(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem,
                                cudaStream_t s);
moe_status_t launch_chain_plain_a(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem,
                                  cudaStream_t s);
moe_status_t launch_chain_plain_b(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem,
                                  cudaStream_t s);

}  // namespace gemm
}  // namespace moe

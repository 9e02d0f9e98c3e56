// S4-S6: grouped block-scaled NVFP4 GEMMs on the fifth-generation tensor core.
//
// Sources: FlashInfer flashinfer.fused_moe.CudnnGroupedGemmNvfp4Config (grouped GEMM1 /
// GEMM2 over expert segments padded to 128 rows; GEMM1 rows times the expert's global
// dequant; the BF16 intermediate quantised to NVFP4 straight into GEMM2's layout; GEMM2's
// global dequant applied to the rows); Megatron-Core core.inference.moe.flashinfer_nvfp4
// (SwiGLU and squared-ReLU experts, per-token activation scale, fc2_input_scale);
// FlashInfer flashinfer.fused_moe.alphamoe_nvfp4_aligned_moe (capacity-sized grid that
// skips work past the device-side valid extent).
//
// One persistent CTA per SM, 320 threads:
//   warp 0       producer: per stage, two 2D TMA tile loads (A: 128 rows x 128 B, B: 256
//                rows x 128 B, 128-byte swizzle) and three 2 KB bulk copies of 128x4 scale
//                tiles, all completing on the stage's full barrier;
//   warp 1       TMEM owner and MMA issuer: per stage, 12 tcgen05.cp of scale tiles into
//                TMEM and 8 tcgen05.mma.kind::mxf4nvf4 (M=128, N=128, K=64, E2M1 x E2M1
//                with UE4M3 scales per 16 values, FP32 accumulation in TMEM);
//   warps 2..9   epilogue: two warps per TMEM lane quarter, one per column half; each pulls
//                its 128 accumulator columns into registers (tcgen05.ld) and releases the
//                accumulator at once, so the next tile's MMAs overlap its scaling,
//                activation and NVFP4 requantisation (GEMM1) or BF16 rows (GEMM2); warps
//                whose 32 rows are all padding skip the arithmetic.
// A work unit is (expert e, 256-column tile nt, 128-row tile mi); units are numbered
// expert-major, then column tile, then row tile, and claimed in that order from an atomic
// counter by whichever CTA's producer is free, so the row tiles of one expert stream the
// same weight tile at the same time and share it in L2. The producer hands each claimed id
// to the MMA and epilogue warps through a 4-entry shared-memory ring. The unit count comes
// from padded_offsets on the device.
// TMEM: columns [0, 256) accumulator (two N=128 halves), [256, 448) scale tiles of the four
// stages (16 columns of A scales + 32 of B scales each). Every wait is bounded.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "host_util.h"
#include "layout.h"

namespace moe {
namespace {

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
constexpr int kThreads = 320;  // producer, MMA, 8 epilogue warps
constexpr int kEpiThreads = 256;
constexpr int kSmemExtra = 1024 /*align*/ + 256 /*barriers*/;
constexpr int kUnitRing = 4;      // work-unit ids handed from the producer to the other roles
constexpr int kRingConsumers = 1 + kEpiThreads / 32;  // MMA thread + one lane per epilogue warp

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

struct GemmParams {
  CUtensorMap tmap_a;     // 128-row activation boxes
  CUtensorMap tmap_a32;   // 32-row boxes, for tiles whose real rows all lie in the first 32
  CUtensorMap tmap_b;
  const uint8_t* sfa;
  const uint8_t* sfb;
  const int32_t* padded_offsets;
  const int32_t* row_to_slot;
  const float* xs;
  const float* alpha;
  void* out;
  uint8_t* out_sf;
  int32_t* dev_status;
  int32_t* tile_counter;  // zeroed before the launch (by the permute kernel)
  int32_t El, Kp, nkb, N, Np, n_tiles, top_k, inter, gated;
  float g2;
};

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
template <int MODE>
__device__ __forceinline__ void load_acc(const GemmParams& p, uint32_t tmem_row, int half, uint32_t* r,
                                         uint64_t* acc_empty) {
  if (MODE != kG2Rows && p.gated) {
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

__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float* v) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

template <int MODE>
__device__ __forceinline__ void epilogue_compute(const GemmParams& p, uint32_t* r, int half, int e, int nt,
                                                 int64_t prow, int slot, float xs_t) {
  const bool real = slot >= 0;
  if constexpr (MODE == kG2Rows) {
    const float d2 = __fmul_rn(p.alpha[e], __fdiv_rn(1.0f, p.g2));
    const int col0 = nt * kTileN + half * 128;
    if (!real || col0 >= p.N) return;
    uint16_t* orow = static_cast<uint16_t*>(p.out) + prow * p.N + col0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(__uint_as_float(r[32 * c + i]), d2);
      store_bf16x32(orow + 32 * c, v);
    }
  } else {
    if (!real) return;
    const float a1 = p.alpha[e];
    const int I = p.inter;
    const int ip16 = static_cast<int>(roundup64(I, kTileK) / 16);  // scale columns of the intermediate
    // intermediate columns [i0, i0 + nout) come from this thread's registers
    const int i0 = p.gated ? nt * 128 + half * 64 : nt * kTileN + half * 128;
    const int nout = p.gated ? 64 : 128;
    if (i0 >= I) return;
    if constexpr (MODE == kG1Preact) {
      const int ld = p.gated ? 2 * I : I;
      float* o = static_cast<float*>(p.out) + prow * ld;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        const float y = __fmul_rn(__fmul_rn(__uint_as_float(r[i]), xs_t), a1);
        if (i < nout) o[i0 + i] = y;                    // gate (or all) columns
        else if (p.gated) o[I + i0 + i - 64] = y;       // up columns
      }
      return;
    }
    // activation, 32 intermediate values at a time
    uint32_t sfw = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c * 32 >= nout) break;
      float h[32];
      if (p.gated) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float yg = __fmul_rn(__fmul_rn(__uint_as_float(r[32 * c + i]), xs_t), a1);
          const float yu = __fmul_rn(__fmul_rn(__uint_as_float(r[64 + 32 * c + i]), xs_t), a1);
          h[i] = bf16_round_f32(__fmul_rn(silu_f32(yg), yu));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float y = fmaxf(__fmul_rn(__fmul_rn(__uint_as_float(r[32 * c + i]), xs_t), a1), 0.0f);
          h[i] = bf16_round_f32(__fmul_rn(y, y));
        }
      }
      const int ic = i0 + 32 * c;
      if constexpr (MODE == kG1Act) {
        store_bf16x32(static_cast<uint16_t*>(p.out) + prow * I + ic, h);
      } else {
        uint8_t* dst = static_cast<uint8_t*>(p.out) + prow * (I / 2) + ic / 2;
        const uint32_t q2 = requant32_store(h, p.g2, dst);
        // two 32-value chunks make one 4-scale group of the 128x4 tile layout
        if (c & 1) {
          *reinterpret_cast<uint32_t*>(p.out_sf + sf_tile_offset(prow, (ic >> 4) - 2, ip16)) = sfw | (q2 << 16);
        } else {
          sfw = q2;
        }
      }
    }
    if constexpr (MODE == kG1Fused) {
      // zero the scale columns of the K padding once per row (last column tile, first half)
      if (nt == p.n_tiles - 1 && half == 0) {
        for (int c4 = I / 64; c4 < ip16 / 4; ++c4)
          *reinterpret_cast<uint32_t*>(p.out_sf + sf_tile_offset(prow, 4 * c4, ip16)) = 0u;
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* final_bar = acc_empty + 1;
  uint64_t* unit_full = final_bar + 1;
  uint64_t* unit_empty = unit_full + kUnitRing;
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(unit_empty + kUnitRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(unit_empty + kUnitRing) + kUnitRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiThreads);
    mbar_init(final_bar, 1);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&unit_full[i], 1);
      mbar_init(&unit_empty[i], kRingConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.tmap_a);
    prefetch_tensormap(&p.tmap_a32);
    prefetch_tensormap(&p.tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();  // the plan, activations and tile counter come from earlier kernels
  for (int i = threadIdx.x; i <= p.El; i += blockDim.x) s_off[i] = p.padded_offsets[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total_units = (s_off[p.El] >> 7) * p.n_tiles;
  // the producer claims work units and hands their ids to the MMA and epilogue warps
  auto take_unit = [&](uint32_t& rslot, uint32_t& rphase, bool one_lane) -> int {
    bool got = mbar_wait(&unit_full[rslot], rphase, abort_flag, p.dev_status);
    if (!one_lane) got = __all_sync(0xffffffffu, got);
    if (!got) return -2;
    const int u = unit_ring[rslot];
    if (!one_lane) __syncwarp();
    if (one_lane || lane == 0) mbar_arrive(&unit_empty[rslot]);
    if (++rslot == kUnitRing) { rslot = 0; rphase ^= 1; }
    return u;
  };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      uint32_t rslot = 0, rphase = 0;
      bool ok = true;
      while (ok) {
        // claim the next unit (in order, from the global counter) and publish its id
        if (!mbar_wait(&unit_empty[rslot], rphase ^ 1, abort_flag, p.dev_status)) { ok = false; break; }
        int u = atomicAdd(p.tile_counter, 1);
        if (u >= total_units) u = -1;
        unit_ring[rslot] = u;
        mbar_arrive(&unit_full[rslot]);
        if (++rslot == kUnitRing) { rslot = 0; rphase ^= 1; }
        if (u < 0) break;
        int e, nt, mi;
        decode_unit(u, s_off, p.El, p.n_tiles, e, nt, mi);
        const int row0 = s_off[e] + mi * kTileM;
        const int brow0 = e * p.Np + nt * kTileN;
        const int64_t kt = p.Kp >> 6;  // 512-byte scale tiles per 128 rows
        const uint8_t* sfa = p.sfa + static_cast<int64_t>(row0 >> 7) * kt * 512;
        const uint8_t* sfb0 = p.sfb + (static_cast<int64_t>(e) * (p.Np >> 7) + nt * 2) * kt * 512;
        const uint8_t* sfb1 = sfb0 + kt * 512;
        // a tile whose row 32 is padding has all its real rows in the first 32 (padding rows
        // end a segment): load only those; the MMA rows fed by stale shared memory are
        // padding rows, whose results are never stored
        const bool short_tile = p.row_to_slot[row0 + 32] < 0;
        const uint32_t tx = short_tile ? kStageTx - (kABytes - 32 * 128) : kStageTx;
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.dev_status)) { ok = false; break; }
          uint8_t* st = smem + stage * kStageBytes;
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_2d(st, short_tile ? &p.tmap_a32 : &p.tmap_a, kb * 128, row0, &full[stage]);
          tma_load_2d(st + kOffB, &p.tmap_b, kb * 128, brow0, &full[stage]);
          bulk_load(st + kOffSfa, sfa + kb * 2048, 2048, &full[stage]);
          bulk_load(st + kOffSfb, sfb0 + kb * 2048, 2048, &full[stage]);
          bulk_load(st + kOffSfb + 2048, sfb1 + kb * 2048, 2048, &full[stage]);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // copies may still be landing in shared memory: let them finish before exit
        for (int s = 0; s < kStages; ++s)
          if (issued_mask & (1u << s)) mbar_drain(&full[s], (issued_phase >> s) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_mxf4nvf4(kTileM, 128);
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      uint32_t rslot = 0, rphase = 0;
      bool ok = true;
      while (ok) {
        const int u = take_unit(rslot, rphase, true);
        if (u < 0) break;
        if (!mbar_wait(acc_empty, acc_phase ^ 1, abort_flag, p.dev_status)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.dev_status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * kStageBytes);
          const uint32_t sft = tmem + kSfCol0 + stage * kSfColsPerStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tmem_cp_sf_tile(sft + kk * 4, sdesc_sf_tile(st + kOffSfa + kk * 512));
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tmem_cp_sf_tile(sft + 16 + h * 16 + kk * 4, sdesc_sf_tile(st + kOffSfb + h * 2048 + kk * 512));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = sdesc_kmajor_sw128(st + kk * 32);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t bdesc = sdesc_kmajor_sw128(st + kOffB + h * (128 * 128) + kk * 32);
              mma_mxf4nvf4(tmem + h * 128, adesc, bdesc, idesc, sft + kk * 4, sft + 16 + h * 16 + kk * 4,
                           (kb | kk) != 0);
            }
          }
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
  } else {
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;       // column half of the tile
    const int r = q * 32 + lane;            // row inside the 128-row tile
    const uint32_t tmem_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t acc_phase = 0;
    uint32_t rslot = 0, rphase = 0;
    while (true) {
      const int u = take_unit(rslot, rphase, false);
      if (u < 0) break;
      int e, nt, mi;
      decode_unit(u, s_off, p.El, p.n_tiles, e, nt, mi);
      const int64_t prow = s_off[e] + mi * kTileM + r;
      const int slot = p.row_to_slot[prow];
      const float xs_t = (MODE != kG2Rows && slot >= 0) ? p.xs[slot / p.top_k] : 0.0f;
      bool ok = mbar_wait(acc_full, acc_phase, abort_flag, p.dev_status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t acc[128];
      load_acc<MODE>(p, tmem_row, half, acc, acc_empty);
      acc_phase ^= 1;
      if (__any_sync(0xffffffffu, slot >= 0)) epilogue_compute<MODE>(p, acc, half, e, nt, prow, slot, xs_t);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // the driver entry point is looked up once per process; it holds no device state
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2D uint8 map over `rows` rows of `row_bytes` bytes, box = 128 bytes x box_rows, 128B swizzle.
// Columns past row_bytes and rows past `rows` read as zero.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
moe_status_t launch_mode(const GemmParams& prm, int64_t units_max, size_t smem, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<MODE>;
  MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
  // persistent: one CTA per SM, at most one per work unit
  const int grid = static_cast<int>(units_max < num_sms() ? units_max : num_sms());
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, prm);
}

}  // namespace

moe_status_t launch_gemm(const GemmLaunch& g, cudaStream_t s) {
  if (g.cap == 0) return MOE_OK;
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  if (!encode_rows(&prm.tmap_a, g.a, g.K / 2, g.cap, kTileM)) return MOE_ERR_CUDA;
  if (!encode_rows(&prm.tmap_a32, g.a, g.K / 2, g.cap, 32)) return MOE_ERR_CUDA;
  if (!encode_rows(&prm.tmap_b, g.b, g.K / 2, g.El * g.Np, kTileN)) return MOE_ERR_CUDA;
  prm.sfa = g.a_sf;
  prm.sfb = g.b_sf;
  prm.padded_offsets = g.padded_offsets;
  prm.row_to_slot = g.row_to_slot;
  prm.xs = g.xs;
  prm.alpha = g.alpha;
  prm.out = g.out;
  prm.out_sf = g.out_sf;
  prm.dev_status = g.dev_status;
  prm.tile_counter = g.tile_counter;
  prm.El = static_cast<int32_t>(g.El);
  prm.Kp = static_cast<int32_t>(g.Kp);
  prm.nkb = static_cast<int32_t>(g.Kp / kTileK);
  prm.N = static_cast<int32_t>(g.N);
  prm.Np = static_cast<int32_t>(g.Np);
  prm.n_tiles = static_cast<int32_t>(g.Np / kTileN);
  prm.top_k = g.top_k;
  prm.inter = g.inter;
  prm.gated = g.gated ? 1 : 0;
  prm.g2 = g.g2;
  const int64_t units_max = (g.cap / kTileM) * prm.n_tiles;
  const size_t smem = static_cast<size_t>(kStages) * kStageBytes + kSmemExtra + (g.El + 1) * 4;
  switch (g.mode) {
    case kG1Fused: return launch_mode<kG1Fused>(prm, units_max, smem, s);
    case kG1Preact: return launch_mode<kG1Preact>(prm, units_max, smem, s);
    case kG1Act: return launch_mode<kG1Act>(prm, units_max, smem, s);
    case kG2Rows: return launch_mode<kG2Rows>(prm, units_max, smem, s);
    default: return MOE_ERR_INVALID_ARGUMENT;
  }
}

}  // namespace moe

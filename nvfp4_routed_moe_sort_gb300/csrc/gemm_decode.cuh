// Decode-shaped grouped GEMMs: GEMM1 and GEMM2 chained in one launch with the operands
// swapped. When every expert holds at most 16 token rows (batches of at most 16 tokens),
// a 128-row activation tile would be almost all padding; here the weight tile is the MMA's
// M = 128 operand (two of them per 256-row weight tile) and the expert's token rows are its
// N = 16 operand, so every TMEM lane of the accumulator is a real output feature and each
// epilogue thread finishes one feature (GEMM1: its gate and up values) for all the tokens.
//
// Same sources and arithmetic as the grouped GEMM (gemm_kernel.cuh): per-16 block-scaled
// E2M1 x E2M1 with UE4M3 scales, FP32 accumulation, GEMM1 rows x per-token scale x expert
// alpha (gate rows x gate alpha), the typed activation, BF16 round and NVFP4 requant with
// the static FC2 input scale; GEMM2 x alpha2 / fc2_input_scale into BF16 rows or FP32
// reductions.
//
// One persistent CTA per SM, 320 threads:
//   warp 0     producer: per stage one 2D TMA load of the 256-row weight tile (128 B of K
//              per row), one of the expert's 16 token rows, two 4 KB and one 2 KB bulk
//              copies of scale tiles; 5 stages of 40 KB;
//   warp 1     TMEM owner and MMA issuer: per stage, once its scales are in TMEM, 8
//              tcgen05.mma.kind::mxf4nvf4 (M=128, N=16, K=64) into one of two accumulator
//              buffers (double-buffered: the next unit's MMAs overlap this one's epilogue);
//   warps 2-5  epilogue, one per TMEM lane quarter;
//   warps 6-9  scale writers, one per TMEM lane quarter: per stage, the 12 scale tiles'
//              lines from shared memory into TMEM (tcgen05.st).
// Work units are (active expert, 256-row weight tile): GEMM1's first, then GEMM2's; a GEMM2
// unit waits (bounded) until every GEMM1 unit of its expert has been written, after loading
// or starting its weight tiles.
//
// Scheduling. When the routing ids are given (the one-call path), CTA b's first unit is unit
// b: while the prologue still computes the plan, the CTA finds that unit's expert from the
// routing ids (an input of the step) and loads the unit's first weight stages (the weights
// depend on no earlier kernel), so the weight stream starts during the prologue. After the
// dependency wait the CTA takes the unit by setting its ownership flag, and keeps the loaded
// stages only if the plan confirms the expert. All other units come from one counter. A CTA
// whose counter claim reaches the GEMM2 units first takes every first unit whose flag is
// still clear, so each GEMM2 wait depends only on GEMM1 units held by running CTAs.
#pragma once

#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "host_util.h"
#include "layout.h"

namespace moe {
namespace dgemm {

constexpr int kTokens = 16;                       // MMA N: token rows per expert
constexpr int kStages = 5;
constexpr int kWBytes = 256 * 128;                // weight tile: two 128-row MMA operands
constexpr int kXBytes = kTokens * 128;            // token rows
constexpr int kSfwBytes = 2 * 4 * 512;            // two 128-row scale tiles x 4 K=64 steps
constexpr int kSfxBytes = 4 * 512;
constexpr int kOffX = kWBytes;
constexpr int kOffSfw = kOffX + kXBytes;
constexpr int kOffSfx = kOffSfw + kSfwBytes;
constexpr int kStageBytes = kOffSfx + kSfxBytes;  // 40 KB
// warp 0 producer, warp 1 MMA issuer, warps 2-5 epilogue, warps 6-9 scale writers (each
// warp reaches only the TMEM lane quarter warp % 4, so each role's four warps cover all 128)
constexpr int kThreads = 320;
constexpr int kEpiWarps = 4;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kSfWriter0 = 2 + kEpiWarps;
constexpr int kSfWriters = 4;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 2 * kTokens;             // one accumulator buffer: two halves x 16 columns
constexpr int kSfCol0 = 2 * kAccCols;             // after the two accumulator buffers
constexpr int kSfColsPerStage = 48;               // 2 weight tiles x 16 + 16 for the tokens
constexpr int kUnitRing = 4;
constexpr int kRingConsumers = 1 + kEpiWarps + kSfWriters;
constexpr int kBarBytes = 512;  // barriers, unit ring, TMEM address, flags
constexpr int kSmemExtra = 1024 /*align*/ + kBarBytes;

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
// full, empty, sf_full, pre per stage; acc_full/acc_empty pairs; final; the unit ring's two
// sets; then the ring, the TMEM address, the abort flag and the active-expert count
static_assert((4 * kStages + 5 + 2 * kUnitRing) * 8 + kUnitRing * 4 + 12 <= kBarBytes, "barrier area");
// the 12 scale atoms of a stage (two weight tiles x 4 K=64 steps, then the tokens' 4) are
// contiguous, atom a feeding TMEM columns [4a, 4a+4) of the stage
static_assert(kOffSfx == kOffSfw + 8 * 512 && kSfColsPerStage == 12 * 4, "scale atom order");

// One GEMM of the launch.
struct Phase {
  CUtensorMap tmap_w;    // weight rows of the prepared layout, box 256 rows x 128 B
  CUtensorMap tmap_x;    // token rows in plan order, box 16 rows x 128 B
  const uint8_t* w_raw;  // the rows behind tmap_w (K/2 bytes each), for the L2 prefetch
  const uint8_t* sfw;
  const uint8_t* sfx;
  const float* alpha;
  const float* alpha_gate;
  void* out;
  uint8_t* out_sf;
  int32_t K, Kp, nkb, Nw, Nwp, n_tiles;  // Nw output features (N1 or H), Nwp padded to 256
};

struct Params {
  Phase ph[2];
  const int32_t* padded_offsets;
  const int32_t* row_to_slot;
  const float* xs;
  int32_t* dev_status;
  int32_t* tile_counter;  // zeroed before the launch
  int32_t* e_done;        // per local expert: GEMM1 epilogue warps done (zeroed before the launch)
  int32_t* own;           // ownership flags of units [0, n_static) (zeroed before the launch)
  int32_t* owned;         // count of the flags set (zeroed before the launch)
  int32_t dbg_hooks;      // test build only: bit 0 wrong guesses, bit 1 odd CTAs skip their offered unit
  int32_t n_static;       // statically offered first units (0: every unit from the counter)
  const int32_t* hint_ids;  // routing ids of the step [hint_slots] (read before the wait)
  int32_t hint_mask, hint_off, hint_slots;
  int32_t El, top_k, inter;
  float g2;
  const void* route_w;
  int32_t route_w_dtype;
  float rsf;
  uint64_t wait_ns;       // limit of every bounded wait (kWaitLimitNs unless a test build shortens it)
  int32_t withhold;       // test build only: the first active expert's GEMM1 units never publish
};

__device__ __forceinline__ void red_add_f32(float* out, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(out), "f"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(int32_t* counter, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(counter), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// how long a CTA about to take a GEMM2 unit waits for the offered units' owners
constexpr uint64_t kSweepGraceNs = 20000;

__device__ __forceinline__ int ld_acquire_s32(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

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

__device__ __forceinline__ void prefetch_l2(const uint8_t* ptr, int64_t bytes) {
  for (int64_t o = 0; o < bytes; o += 65536) {
    const int64_t n = bytes - o < 65536 ? bytes - o : 65536;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr + o), "r"(static_cast<uint32_t>(n))
                 : "memory");
  }
}

__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

__device__ __forceinline__ float silu_f32(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }
__device__ __forceinline__ float gelu_f32(float x) {
  return __fmul_rn(__fmul_rn(0.5f, x), __fadd_rn(1.0f, erff(__fmul_rn(x, 0.70710678118654752f))));
}
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
__host__ __device__ constexpr bool gated_act(int act) { return act == MOE_ACT_SWIGLU || act == MOE_ACT_GEGLU; }

// Requantise one value per lane: 16 consecutive lanes hold one 16-value block (16
// consecutive intermediate features of one token). Every lane of the warp must call it.
// The arithmetic is the block rule of quantize_block16.
__device__ __forceinline__ void requant_lanes(float h, bool store, float g2, int lane, uint8_t* code_byte,
                                              uint8_t* scale_byte) {
  float amax = fmaxf(0.0f, fabsf(h));
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  const float sc = __fmul_rn(__fdiv_rn(amax, 6.0f), g2);
  const uint32_t qs = f32_to_e4m3(sc);
  const float qf = e4m3_to_f32(qs);
  const float inv = (qf == 0.0f) ? 0.0f : __fdiv_rn(g2, qf);
  const float hn = __shfl_down_sync(0xffffffffu, h, 1);
  if (store) {
    if ((lane & 1) == 0) *code_byte = static_cast<uint8_t>(f32x2_to_e2m1(__fmul_rn(h, inv), __fmul_rn(hn, inv)));
    if ((lane & 15) == 0) *scale_byte = static_cast<uint8_t>(qs);
  }
}

// ROWS: GEMM2 writes BF16 rows (true) or adds route-weighted rows into FP32 (false).
template <bool ROWS, int ACT>
__global__ void __launch_bounds__(kThreads, 1) decode_gemm_kernel(const __grid_constant__ Params p) {
  constexpr bool kGated = gated_act(ACT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;   // [2]
  uint64_t* acc_empty = acc_full + 2;     // [2]
  uint64_t* final_bar = acc_empty + 2;
  uint64_t* unit_full = final_bar + 1;
  uint64_t* unit_empty = unit_full + kUnitRing;
  uint64_t* pre_bar = unit_empty + kUnitRing;  // [kStages] weight stages loaded before the wait
  uint64_t* sf_full = pre_bar + kStages;       // [kStages] the stage's scales are in TMEM
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(sf_full + kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + kStages) + kUnitRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_nact = const_cast<int*>(abort_flag) + 1;
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + kBarBytes);
  int32_t* s_act = s_off + roundup64(p.El + 1, 4);  // active local experts, ascending
  uint8_t* s_flag = reinterpret_cast<uint8_t*>(s_act + p.El);  // routed local experts (from the ids)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiThreads);
    }
    for (int s = 0; s < kStages; ++s) mbar_init(&pre_bar[s], 1);
    for (int s = 0; s < kStages; ++s) mbar_init(&sf_full[s], kSfWriters);
    mbar_init(final_bar, 1);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&unit_full[i], 1);
      mbar_init(&unit_empty[i], kRingConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 2; ++i) {
      prefetch_tensormap(&p.ph[i].tmap_w);
      prefetch_tensormap(&p.ph[i].tmap_x);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // The first unit's weight stages, before the wait (see the scheduling note above): the
  // routed local experts from the ids, the expert ranked blockIdx.x / n_tiles among them.
  int pre_n = 0, pre_e = -1;  // (producer thread) stages loaded, their expert
  if (warp == 0 && static_cast<int>(blockIdx.x) < p.n_static) {
    for (int i = lane; i < p.El; i += 32) s_flag[i] = 0;
    __syncwarp();
    for (int i = lane; i < p.hint_slots; i += 32) {
      const int l = (p.hint_ids[i] & p.hint_mask) - p.hint_off;
      if (l >= 0 && l < p.El) s_flag[l] = 1;
    }
    __syncwarp();
    const int want = static_cast<int>(blockIdx.x) / p.ph[0].n_tiles + (p.dbg_hooks & 1);
    int n = 0, e_first = -1;
    for (int base = 0; base < p.El && n <= want; base += 32) {
      const int l = base + lane;
      const bool act = l < p.El && s_flag[l] != 0;
      const unsigned ball = __ballot_sync(0xffffffffu, act);
      if (act && n + __popc(ball & ((1u << lane) - 1u)) == want) e_first = l;
      n += __popc(ball);
    }
    e_first = __reduce_max_sync(0xffffffffu, e_first);
    if (lane == 0 && e_first >= 0) {
      const Phase& ph = p.ph[0];
      const int nt = static_cast<int>(blockIdx.x) % ph.n_tiles;
      const int wrow0 = e_first * ph.Nwp + nt * 256;
      const int64_t kt = ph.Kp >> 6;
      const uint8_t* sfw0 = ph.sfw + (static_cast<int64_t>(e_first) * (ph.Nwp >> 7) + nt * 2) * kt * 512;
      const uint8_t* sfw1 = sfw0 + kt * 512;
      pre_n = ph.nkb < kStages ? ph.nkb : kStages;
      pre_e = e_first;
      for (int kb = 0; kb < pre_n; ++kb) {
        uint8_t* st = smem + kb * kStageBytes;
        mbar_arrive_expect_tx(&pre_bar[kb], kWBytes + kSfwBytes);
        tma_load_2d(st, &ph.tmap_w, kb * 128, wrow0, &pre_bar[kb]);
        bulk_load(st + kOffSfw, sfw0 + kb * 2048, 2048, &pre_bar[kb]);
        bulk_load(st + kOffSfw + 2048, sfw1 + kb * 2048, 2048, &pre_bar[kb]);
      }
    }
  }
  pdl_wait();  // the plan, the token rows and the counters come from earlier kernels
  // the producer's claim of its offered unit goes out now; its round trip overlaps the
  // plan load below (whether the unit is offered at all is known only after it)
  int cas_old = 1;
  int next_claim = 0;  // the producer's counter claim for its next unit, issued one unit early
  if (threadIdx.x == 0) {
    if (static_cast<int>(blockIdx.x) < p.n_static && !((p.dbg_hooks & 2) && (blockIdx.x & 1)))
      cas_old = atomicCAS(p.own + blockIdx.x, 0, 1);
    next_claim = atomicAdd(p.tile_counter, 1);
  }
  for (int i = threadIdx.x; i <= p.El; i += blockDim.x) s_off[i] = p.padded_offsets[i];
  __syncthreads();
  if (warp == 0) {
    // compact the active experts (non-empty segments), in ascending order
    int n = 0;
    for (int base = 0; base < p.El; base += 32) {
      const int l = base + lane;
      const bool act = l < p.El && s_off[l + 1] > s_off[l];
      const unsigned ball = __ballot_sync(0xffffffffu, act);
      if (act) s_act[n + __popc(ball & ((1u << lane) - 1u))] = l;
      n += __popc(ball);
    }
    if (lane == 0) *s_nact = n;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_active = *s_nact;
  const int units0 = n_active * p.ph[0].n_tiles;
  const int total_units = units0 + n_active * p.ph[1].n_tiles;
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

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      uint32_t rslot = 0, rphase = 0;
      bool ok = true;
      // units [0, n_first) are offered to CTAs 0..n_first-1 (GEMM1 units only), the rest
      // come from the counter
      const int n_first = p.n_static < units0 ? p.n_static : units0;
      const int u_static = static_cast<int>(blockIdx.x) < n_first ? static_cast<int>(blockIdx.x) : -1;
      int u_held = -1;  // a counter claim kept while the offered units are swept
      int sweep = 0;    // next offered unit to check before the first GEMM2 unit
      bool first = true;
      while (ok) {
        if (!mbar_wait(&unit_empty[rslot], rphase ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
        int u = -1;
        if (first) {
          first = false;
          // the claim issued after the wait (flags past the offered range are never read)
          if (u_static >= 0 && cas_old == 0) {
            u = u_static;
            atomicAdd(p.owned, 1);
          }
        }
        while (u < 0) {
          if (u_held < 0) {
            // the claim issued one unit ago; the next one goes out now, so its round trip
            // overlaps this unit's loads
            u_held = n_first + next_claim;
            next_claim = atomicAdd(p.tile_counter, 1);
            if (u_held < units0) {  // GEMM1 units need no sweep
              u = u_held;
              u_held = -1;
              break;
            }
          }
          // before any GEMM2 unit (or the end): every offered unit is owned by a running CTA.
          // Normally all are by now (one load); late owners get a grace period, then the
          // units still free are taken here.
          if (sweep < n_first) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_s32(p.owned) < n_first && globaltimer_ns() - t0 < kSweepGraceNs) __nanosleep(128);
            if (ld_acquire_s32(p.owned) >= n_first) sweep = n_first;
          }
          while (sweep < n_first && u < 0) {
            if (__ldcg(p.own + sweep) == 0 && atomicCAS(p.own + sweep, 0, 1) == 0) {
              u = sweep;
              atomicAdd(p.owned, 1);
            }
            ++sweep;
          }
          if (u >= 0) break;
          u = u_held < total_units ? u_held : -1;
          u_held = -1;
          break;
        }
        unit_ring[rslot] = u;
        mbar_arrive(&unit_full[rslot]);
        if (++rslot == kUnitRing) { rslot = 0; rphase ^= 1; }
        if (pre_n > 0) {
          // the stages loaded before the wait land before their buffers are reused
          for (int kb = 0; kb < pre_n; ++kb)
            if (!mbar_wait(&pre_bar[kb], 0, abort_flag, p.dev_status, p.wait_ns)) ok = false;
          if (!ok) break;
        }
        if (u < 0) break;
        const bool second = u >= units0;
        const Phase& ph = p.ph[second ? 1 : 0];
        const int uu = second ? u - units0 : u;
        const int e = s_act[uu / ph.n_tiles], nt = uu % ph.n_tiles;
        const int seg = s_off[e];
        const int wrow0 = e * ph.Nwp + nt * 256;
        const int64_t kt = ph.Kp >> 6;  // 512-byte scale tiles per 128 rows
        const uint8_t* sfw0 = ph.sfw + (static_cast<int64_t>(e) * (ph.Nwp >> 7) + nt * 2) * kt * 512;
        const uint8_t* sfw1 = sfw0 + kt * 512;
        const uint8_t* sfx = ph.sfx + static_cast<int64_t>(seg >> 7) * kt * 512;
        // A GEMM2 unit depends on every GEMM1 unit of its expert, its weights do not. When
        // the unit fits in the pipeline, its weight tiles are loaded first, then the wait,
        // then the token rows (each stage's barrier expects both parts); otherwise the
        // weight tile is started towards L2 before the wait.
        int pre = 0;
        uint32_t pre_stage = stage;
        if (pre_n > 0) {
          // this CTA's first unit: keep the weight stages loaded before the wait if the plan
          // confirms their expert, else reload them in full below
          if (u == u_static && !second && e == pre_e) {
            for (int kb = 0; kb < pre_n; ++kb) {
              if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
              uint8_t* st = smem + stage * kStageBytes;
              mbar_arrive_expect_tx(&full[stage], kXBytes + kSfxBytes);
              tma_load_2d(st + kOffX, &ph.tmap_x, kb * 128, seg, &full[stage]);
              bulk_load(st + kOffSfx, sfx + kb * 2048, 2048, &full[stage]);
              issued_mask |= 1u << stage;
              issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
              if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            pre = pre_n;
          }
          pre_n = 0;
        }
        if (second && ph.nkb > kStages) {
          const int target = kEpiWarps * p.ph[0].n_tiles;
          if (ld_acquire_s32(p.e_done + e) < target) {  // only a unit that will wait prefetches
            prefetch_l2(ph.w_raw + static_cast<int64_t>(wrow0) * (ph.K / 2), static_cast<int64_t>(256) * (ph.K / 2));
            prefetch_l2(sfw0, 2 * kt * 512);
            if (!wait_counter(p.e_done + e, target, abort_flag, p.dev_status, p.wait_ns)) {
              ok = false;
              break;
            }
          }
          fence_proxy_async_global();  // the TMA reads below follow the observed generic writes
        } else if (second) {
          pre = ph.nkb;
          for (int kb = 0; kb < pre; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
            uint8_t* st = smem + stage * kStageBytes;
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            tma_load_2d(st, &ph.tmap_w, kb * 128, wrow0, &full[stage]);
            bulk_load(st + kOffSfw, sfw0 + kb * 2048, 2048, &full[stage]);
            bulk_load(st + kOffSfw + 2048, sfw1 + kb * 2048, 2048, &full[stage]);
            issued_mask |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          if (!wait_counter(p.e_done + e, kEpiWarps * p.ph[0].n_tiles, abort_flag, p.dev_status, p.wait_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();  // the TMA reads below follow the observed generic writes
          for (int kb = 0; kb < pre; ++kb) {
            uint8_t* st = smem + pre_stage * kStageBytes;
            tma_load_2d(st + kOffX, &ph.tmap_x, kb * 128, seg, &full[pre_stage]);
            bulk_load(st + kOffSfx, sfx + kb * 2048, 2048, &full[pre_stage]);
            if (++pre_stage == kStages) pre_stage = 0;
          }
        }
        for (int kb = pre; kb < ph.nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
          uint8_t* st = smem + stage * kStageBytes;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          tma_load_2d(st, &ph.tmap_w, kb * 128, wrow0, &full[stage]);
          tma_load_2d(st + kOffX, &ph.tmap_x, kb * 128, seg, &full[stage]);
          bulk_load(st + kOffSfw, sfw0 + kb * 2048, 2048, &full[stage]);
          bulk_load(st + kOffSfw + 2048, sfw1 + kb * 2048, 2048, &full[stage]);
          bulk_load(st + kOffSfx, sfx + kb * 2048, 2048, &full[stage]);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // every issued copy lands before the CTA exits (after an abort, or when another role
      // gave up before consuming it)
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) mbar_drain(&full[s], (issued_phase >> s) & 1);
      for (int kb = 0; kb < pre_n; ++kb) mbar_drain(&pre_bar[kb], 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_mxf4nvf4(128, kTokens);
      uint32_t stage = 0, phase = 0, buf = 0;
      uint32_t acc_phase[2] = {0, 0};
      uint32_t rslot = 0, rphase = 0;
      bool ok = true;
      while (ok) {
        const int u = take_unit(rslot, rphase, true);
        if (u < 0) break;
        if (!mbar_wait(&acc_empty[buf], acc_phase[buf] ^ 1, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const int nkb = p.ph[u >= units0 ? 1 : 0].nkb;
        const uint32_t acc = tmem + buf * kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          // the stage has landed and the writer warps have put its scales in TMEM: the
          // weight tiles' at [h*16 + kk*4, +4), the tokens' at [32 + kk*4, +4)
          if (!mbar_wait(&sf_full[stage], phase, abort_flag, p.dev_status, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * kStageBytes);
          const uint32_t sft = tmem + kSfCol0 + stage * kSfColsPerStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t xdesc = sdesc_kmajor_sw128(st + kOffX + kk * 32);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t wdesc = sdesc_kmajor_sw128(st + h * (128 * 128) + kk * 32);
              mma_mxf4nvf4(acc + h * kTokens, wdesc, xdesc, idesc, sft + h * 16 + kk * 4, sft + 32 + kk * 4,
                           (kb | kk) != 0);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
        acc_phase[buf] ^= 1;
        buf ^= 1;
      }
      tc_commit(final_bar);
      mbar_drain(final_bar, 0);
    }
  } else if (warp >= kSfWriter0) {
    // Scale writers: per stage, once it has landed, each writer warp stores the stage's 12
    // scale atoms into its own TMEM lane quarter (tcgen05.st), line l of an atom to lane l,
    // as a copy replicated over the four quarters would put it. A stage's scale columns are
    // free once it has landed: the producer reloads a stage only after the MMAs that read it
    // have completed.
    const uint32_t sf_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kSfCol0;
    uint32_t stage = 0, phase = 0;
    uint32_t rslot = 0, rphase = 0;
    bool ok = true;
    while (ok) {
      const int u = take_unit(rslot, rphase, false);
      if (u < 0) break;
      const int nkb = p.ph[u >= units0 ? 1 : 0].nkb;
      for (int kb = 0; kb < nkb; ++kb) {
        const bool got = mbar_wait(&full[stage], phase, abort_flag, p.dev_status, p.wait_ns);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const uint4* atoms = reinterpret_cast<const uint4*>(smem + stage * kStageBytes + kOffSfw);
        const uint32_t sft = sf_lane + stage * kSfColsPerStage;
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 w = atoms[(4 * part + i) * 32 + lane];
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
  } else {
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q * 32 + lane;            // weight row of each 128-row half = output feature
    const uint32_t tmem_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t buf = 0;
    uint32_t acc_phase[2] = {0, 0};
    uint32_t rslot = 0, rphase = 0;
    while (true) {
      const int u = take_unit(rslot, rphase, false);
      if (u < 0) break;
      const bool second = u >= units0;
      const Phase& ph = p.ph[second ? 1 : 0];
      const int uu = second ? u - units0 : u;
      const int e = s_act[uu / ph.n_tiles], nt = uu % ph.n_tiles;
      const int seg = s_off[e];
      // the expert's token rows lead its segment: their slots, per-token scales / weights
      int slot[kTokens];
      float sc[kTokens];
      int n_e = 0;
#pragma unroll
      for (int t = 0; t < kTokens; ++t) {
        slot[t] = (seg + t < s_off[e + 1]) ? p.row_to_slot[seg + t] : -1;
        n_e += slot[t] >= 0 ? 1 : 0;
      }
#pragma unroll
      for (int t = 0; t < kTokens; ++t) {
        sc[t] = 0.0f;
        if (slot[t] >= 0) {
          if (!second)
            sc[t] = p.xs[slot[t] / p.top_k];
          else if constexpr (!ROWS)
            sc[t] = route_weight(p.route_w, p.route_w_dtype, slot[t], p.rsf);
        }
      }
      const float a = ph.alpha[e];
      const float ag = (!second && kGated) ? ph.alpha_gate[e] : a;
      bool ok = mbar_wait(&acc_full[buf], acc_phase[buf], abort_flag, p.dev_status, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[2 * kTokens];  // [half][token]
      tmem_ld16_issue(tmem_lane + buf * kAccCols, v);
      tmem_ld16_issue(tmem_lane + buf * kAccCols + kTokens, v + kTokens);
      tmem_wait_ld<2 * kTokens>(v);
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      acc_phase[buf] ^= 1;
      buf ^= 1;
      if (!second) {
        const int I = p.inter;
        const int ip16 = static_cast<int>(roundup64(I, kTileK) / 16);
        uint8_t* out = static_cast<uint8_t*>(ph.out);
        // gated: feature nt*128 + r from gate half 0 and up half 1; otherwise the two halves
        // are features nt*256 + r and nt*256 + 128 + r
#pragma unroll
        for (int h = 0; h < (kGated ? 1 : 2); ++h) {
          const int ic = kGated ? nt * 128 + r : nt * kTileN + h * 128 + r;
          const bool col_ok = ic < I;  // uniform per warp (I is a multiple of 128)
#pragma unroll
          for (int t = 0; t < kTokens; ++t) {
            if (t >= n_e) break;  // uniform: n_e is the same in every thread
            float hv = 0.0f;
            if (col_ok) {
              const float yg = __fmul_rn(__fmul_rn(__uint_as_float(v[h * kTokens + t]), sc[t]), kGated ? ag : a);
              const float yu = kGated ? __fmul_rn(__fmul_rn(__uint_as_float(v[kTokens + t]), sc[t]), a) : 0.0f;
              hv = bf16_round_f32(activation_f32<ACT>(yg, yu));
            }
            const int64_t prow = seg + t;
            requant_lanes(hv, col_ok, p.g2, lane, out + prow * (I / 2) + ic / 2,
                          ph.out_sf + sf_tile_offset(prow, ic >> 4, ip16));
          }
        }
        // zero the scale columns of the K padding of GEMM2's operand (last weight tile)
        if (nt == ph.n_tiles - 1 && r < ip16 - I / 16)
          for (int t = 0; t < n_e && t < kTokens; ++t) ph.out_sf[sf_tile_offset(seg + t, I / 16 + r, ip16)] = 0;
        // publish this warp's share of the GEMM1 tile to the GEMM2 units of the expert
        __syncwarp();
        if (lane == 0 && !(p.withhold && e == s_act[0])) red_release_add(p.e_done + e, 1);
      } else {
        const float d2 = __fmul_rn(a, __fdiv_rn(1.0f, p.g2));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int col = nt * kTileN + h * 128 + r;
          if (col >= ph.Nw) continue;
#pragma unroll
          for (int t = 0; t < kTokens; ++t) {
            if (t >= n_e) break;
            const float y = __fmul_rn(__uint_as_float(v[h * kTokens + t]), d2);
            if constexpr (ROWS) {
              static_cast<uint16_t*>(ph.out)[static_cast<int64_t>(seg + t) * ph.Nw + col] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(y));
            } else {
              red_add_f32(static_cast<float*>(ph.out) + static_cast<int64_t>(slot[t] / p.top_k) * ph.Nw + col,
                          __fmul_rn(y, sc[t]));
            }
          }
        }
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

template <bool ROWS, int ACT>
moe_status_t launch_kernel(const Params& prm, int grid, size_t smem, cudaStream_t s) {
  auto kern = decode_gemm_kernel<ROWS, ACT>;
  MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, prm);
}

moe_status_t launch_act(bool rows, int act, const Params& prm, int grid, size_t smem, cudaStream_t s);

}  // namespace dgemm
}  // namespace moe

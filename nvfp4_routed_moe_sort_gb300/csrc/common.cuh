// Shared device helpers for the NVFP4 routed-MoE kernels (sm_103a).
//
// Inline PTX wrappers for mbarriers, TMA (bulk and tiled tensor copies) and the
// fifth-generation tensor core (tcgen05: TMEM allocation, block-scaled MMA,
// shared->TMEM copies, TMEM loads), the NVFP4 element conversions, and the
// 128-row x 4-scale tile layout the block-scaled MMA reads its scales from.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_nvfp4.h"

namespace moe {

// ---------------------------------------------------------------------------
// sizes shared by host and device
// ---------------------------------------------------------------------------
constexpr int kSegAlign = 128;     // expert segments padded to 128 rows
constexpr int kBlock = 16;         // NVFP4 block size
constexpr int kTileM = 128;        // GEMM rows per tile (one MMA M)
constexpr int kTileN = 256;        // GEMM columns per tile (one N=256 MMA per K step)
constexpr int kTileK = 256;        // K elements per pipeline stage (128 bytes per row)
constexpr int kMaxLocalExperts = 512;

__host__ __device__ constexpr int64_t roundup64(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Byte offset of scale (row r, scale column c) in a 128x4-tiled scale matrix whose rows are
// padded to 128 and whose scale columns are padded to `kcols_padded` (a multiple of 16, i.e.
// K padded to 256). A tile of 128 rows x 4 scales is 512 contiguous bytes: byte
// (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4. Tiles are ordered row-tile-major, then by
// scale-column group. Line l of a tile (16 bytes: rows l, l+32, l+64, l+96) is what TMEM
// lane l of every lane quarter holds in the scale layout of an M=128 block-scaled MMA (the
// layout a replicating tcgen05.cp.32x128b.warpx4 copy of the tile produces), so the GEMMs
// load a tile with one bulk copy and store its lines into TMEM unchanged.
__host__ __device__ __forceinline__ int64_t sf_tile_offset(int64_t r, int64_t c, int64_t kcols_padded) {
  return ((r >> 7) * (kcols_padded >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// ---------------------------------------------------------------------------
// NVFP4 element conversions (hardware round-to-nearest-even with saturation)
// ---------------------------------------------------------------------------
// float -> float8_e4m3fn byte, RNE, saturating at +-448
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFF;
}

// float8_e4m3fn byte -> float (exact; the byte never encodes NaN here)
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t s = (b & 0x80u) << 24;
  const uint32_t e = (b >> 3) & 0xF;
  const uint32_t m = b & 0x7;
  float v;
  if (e == 0) {
    v = (float)m * 0.001953125f;  // m/8 * 2^-6, exact
  } else {
    v = __uint_as_float(((e + 120u) << 23) | (m << 20));
  }
  return __uint_as_float(__float_as_uint(v) | s);
}

// two floats -> one byte of two E2M1 codes; `lo` goes to the low nibble
__device__ __forceinline__ uint32_t f32x2_to_e2m1(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}\n"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xFF;
}

// Quantise one 16-value block with encode scale g: returns the scale byte, writes 8 code
// bytes (element 2i in the low nibble of byte i) to codes[0..1] as two uint32 words.
// All arithmetic is single IEEE float32 in the order: s = (amax / 6) * g; q = e4m3(s);
// inv = q == 0 ? 0 : g / q; code = e2m1(x * inv).
__device__ __forceinline__ uint32_t quantize_block16(const float* x, float g, uint32_t codes[2]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float s = __fmul_rn(__fdiv_rn(amax, 6.0f), g);
  const uint32_t q = f32_to_e4m3(s);
  const float qf = e4m3_to_f32(q);
  const float inv = (qf == 0.0f) ? 0.0f : __fdiv_rn(g, qf);
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int i = w * 8 + b * 2;
      word |= f32x2_to_e2m1(__fmul_rn(x[i], inv), __fmul_rn(x[i + 1], inv)) << (8 * b);
    }
    codes[w] = word;
  }
  return q;
}

constexpr float kGlobalNumerator = 2688.0f;  // FLOAT8_E4M3_MAX * FLOAT4_E2M1_MAX: g_enc = 2688 / amax

// 16 BF16 values (two 16-byte loads) -> FP32
__device__ __forceinline__ void load_block16(const uint16_t* src, float* v) {
  const uint4 a = *reinterpret_cast<const uint4*>(src);
  const uint4 b = *reinterpret_cast<const uint4*>(src + 8);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Route weight of slot i stored as FP32, BF16 or packed (BF16 score in bits 31..16),
// times the routed scaling factor: fp32(w * rsf).
__device__ __forceinline__ float route_weight(const void* w, int dtype, int64_t i, float rsf) {
  float v;
  if (dtype == MOE_WEIGHTS_F32)
    v = static_cast<const float*>(w)[i];
  else if (dtype == MOE_WEIGHTS_BF16)
    v = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(w)[i]) << 16);
  else
    v = __uint_as_float(static_cast<const uint32_t*>(w)[i] & 0xFFFF0000u);
  return __fmul_rn(v, rsf);
}

__device__ __forceinline__ float bf16_round_f32(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: kernels of the path are launched so that the next one may
// start while this one runs; each kernel lets its dependents launch at entry, does its
// prologue (no global memory), and waits for its predecessor before touching its outputs.
// Without the launch attribute both instructions are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// shared memory, mbarrier, TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A wait that gives up: after `limit_ns` it raises the CTA's abort flag, ORs
// MOE_DEV_TIMEOUT into the status word and returns false. It also returns false as soon as
// another role of the CTA has aborted. The kernels take the limit as a launch parameter:
// kWaitLimitNs from every product entry point.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* dev_status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      if (dev_status) atomicOr(dev_status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// 2D tiled TMA load of box (x = byte column, y = row) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(smem_dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// contiguous bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0)
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (TMEM + block-scaled MMA)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// arrive on `bar` once every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}


// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row groups 1024 bytes apart. `saddr` is the start (the 1024-aligned tile base plus the
// byte offset of the K slice inside the 128-byte row).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);  // start address >> 4          [0, 14)
  d |= (uint64_t)(16 >> 4) << 16;           // leading byte offset (unused) [16, 30)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset           [32, 46)
  d |= (uint64_t)1 << 46;                   // descriptor version           [46, 48)
  d |= (uint64_t)2 << 61;                   // layout: 128-byte swizzle     [61, 64)
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::mxf4nvf4 with E2M1 A and B, K-major both,
// UE4M3 scales, FP32 accumulation, shape M x N (x K=64).
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(int M, int N) {
  return (1u << 7)                              // A format: E2M1
         | (1u << 10)                           // B format: E2M1
         | ((uint32_t)(N >> 3) << 17)           // N / 8
         | (0u << 23)                           // scale format: UE4M3
         | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// D[tmem] (+)= A[smem] x B[smem]^T with per-16 block scales read from TMEM.
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Each thread of the warp loads 32 consecutive 32-bit columns of its TMEM lane into r[].
// The values are valid only after tmem_wait_ld(r...) below.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Each thread of the warp loads 16 consecutive 32-bit columns of its TMEM lane into r[].
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Wait for every tcgen05.ld issued by this thread; the empty asm statements after the wait
// tie the N loaded registers to it so no use of them is scheduled earlier.
template <int N>
__device__ __forceinline__ void tmem_wait_ld(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Each thread of the warp stores 16 consecutive 32-bit columns of its TMEM lane from r[].
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Wait until every tcgen05.st issued by this thread has been performed.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Per-warpgroup register budget: every warp of the warpgroup executes the same call.
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  tmem_ld32_issue(taddr, r);
  tmem_wait_ld<32>(r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe

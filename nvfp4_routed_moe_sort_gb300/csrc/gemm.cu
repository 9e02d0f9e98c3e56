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
// One persistent CTA per SM, 512 threads (setmaxnreg: 184 registers for the epilogue
// warpgroups, 72 for the rest):
//   warp 0       producer: per stage, two 2D TMA tile loads (A: 128 rows x 128 B, B: 256
//                rows x 128 B, 128-byte swizzle) and three 2 KB bulk copies of 128x4 scale
//                tiles, all completing on the stage's full barrier;
//   warp 1       TMEM owner and MMA issuer: per stage, 4 tcgen05.mma.kind::mxf4nvf4 (M=128,
//                N=256, K=64, E2M1 x E2M1 with UE4M3 scales per 16 values, FP32
//                accumulation in TMEM), once the stage's scales are in TMEM;
//   warps 2, 3, 12, 13  scale writers, one per TMEM lane quarter: per stage, the 12 scale
//                tiles' lines from shared memory into TMEM (tcgen05.st);
//   warps 4..11  epilogue: two warps per TMEM lane quarter, one per column half; each pulls
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
// TMEM: columns [0, 256) accumulator, [256, 448) scale tiles of the four stages (16 columns
// of A scales + 32 of B scales each, the B scales of one K step in 8 adjacent columns: the
// 128-row halves side by side, as the N=256 MMA reads them). Every wait is bounded.
#include "gemm_kernel.cuh"
#include "gemm_decode.cuh"

namespace moe {
namespace {

using namespace gemm;

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

}  // namespace

namespace gemm {

bool fill_phase(Phase& ph, const GemmLaunch& g) {
  if (!encode_rows(&ph.tmap_a, g.a, g.K / 2, g.cap, kTileM)) return false;
  if (!encode_rows(&ph.tmap_a32, g.a, g.K / 2, g.cap, 32)) return false;
  if (!encode_rows(&ph.tmap_b, g.b, g.K / 2, g.El * g.Np, kTileN)) return false;
  ph.b_raw = g.b;
  ph.sfa = g.a_sf;
  ph.sfb = g.b_sf;
  ph.alpha = g.alpha;
  ph.alpha_gate = g.alpha_gate;
  ph.out = g.out;
  ph.out_sf = g.out_sf;
  // rows are N (a multiple of 128) BF16 values long and stored from 32-value column offsets,
  // so a 32-byte aligned base keeps every row store 32-byte aligned
  ph.out_v8 = (reinterpret_cast<uintptr_t>(g.out) & 31) == 0;
  ph.K = static_cast<int32_t>(g.K);
  ph.Kp = static_cast<int32_t>(g.Kp);
  ph.nkb = static_cast<int32_t>(g.Kp / kTileK);
  ph.N = static_cast<int32_t>(g.N);
  ph.Np = static_cast<int32_t>(g.Np);
  ph.n_tiles = static_cast<int32_t>(g.Np / kTileN);
  return true;
}

void fill_common(GemmParams& prm, const GemmLaunch& g) {
  prm.padded_offsets = g.padded_offsets;
  prm.row_to_slot = g.row_to_slot;
  prm.xs = g.xs;
  prm.dev_status = g.dev_status;
  prm.tile_counter = g.tile_counter;
  prm.El = static_cast<int32_t>(g.El);
  prm.top_k = g.top_k;
  prm.inter = g.inter;
  prm.gated = g.gated ? 1 : 0;
  prm.act = g.act;
  prm.g2 = g.g2;
  prm.route_w = g.route_w;
  prm.route_w_dtype = g.route_w_dtype;
  prm.rsf = g.rsf;
}

size_t smem_bytes(int64_t El, bool sparse) {
  return static_cast<size_t>(kStages) * kStageBytes + kSmemExtra + roundup64((El + 1) * 4, 16) +
         (sparse ? kSparseStageBytes : 0);
}

}  // namespace gemm

namespace {

moe_status_t dispatch_chain(int mode, int act, const GemmParams& prm, int64_t units_max, size_t smem,
                            cudaStream_t s) {
  switch (act) {
    case MOE_ACT_SWIGLU:
    case MOE_ACT_GEGLU: return gemm::launch_chain_gated(mode, act, prm, units_max, smem, s);
    case MOE_ACT_RELU2:
    case MOE_ACT_GELU:
    case MOE_ACT_RELU: return gemm::launch_chain_plain_a(mode, act, prm, units_max, smem, s);
    case MOE_ACT_SILU:
    case MOE_ACT_IDENTITY: return gemm::launch_chain_plain_b(mode, act, prm, units_max, smem, s);
    default: return MOE_ERR_INVALID_ARGUMENT;
  }
}

}  // namespace

moe_status_t launch_gemm_chain(const GemmLaunch& g1, const GemmLaunch& g2, int32_t* mt_done, const TestOptions& topt,
                               cudaStream_t s) {
  if (g1.cap == 0) return MOE_OK;
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  if (!fill_phase(prm.ph[0], g1) || !fill_phase(prm.ph[1], g2)) return MOE_ERR_CUDA;
  fill_common(prm, g1);
  prm.route_w = g2.route_w;  // the combine scalars are GEMM2's
  prm.route_w_dtype = g2.route_w_dtype;
  prm.rsf = g2.rsf;
  prm.mt_done = mt_done;
  prm.sparse = g1.El <= kSparseMaxExperts;
  prm.wait_ns = topt.wait_limit_ns;
  prm.withhold = topt.withhold_release;
  const int mode = g2.mode == kG2Reduce ? kChainReduce : kChainRows;
  const int64_t units_max = (g1.cap / kTileM) * (prm.ph[0].n_tiles + prm.ph[1].n_tiles);
  return dispatch_chain(mode, g1.act, prm, units_max, smem_bytes(g1.El, prm.sparse), s);
}

moe_status_t launch_gemm_decode(const GemmLaunch& g1, const GemmLaunch& g2, int32_t* e_done, int32_t* own,
                                const RoutingHint& hint, const TestOptions& topt, cudaStream_t s) {
  if (g1.cap == 0) return MOE_OK;
  dgemm::Params prm;
  memset(&prm, 0, sizeof(prm));
  const GemmLaunch* gs[2] = {&g1, &g2};
  for (int i = 0; i < 2; ++i) {
    const GemmLaunch& g = *gs[i];
    dgemm::Phase& ph = prm.ph[i];
    if (!encode_rows(&ph.tmap_w, g.b, g.K / 2, g.El * g.Np, kTileN)) return MOE_ERR_CUDA;
    if (!encode_rows(&ph.tmap_x, g.a, g.K / 2, g.cap, dgemm::kTokens)) return MOE_ERR_CUDA;
    ph.w_raw = g.b;
    ph.sfw = g.b_sf;
    ph.sfx = g.a_sf;
    ph.alpha = g.alpha;
    ph.alpha_gate = g.alpha_gate;
    ph.out = g.out;
    ph.out_sf = g.out_sf;
    ph.K = static_cast<int32_t>(g.K);
    ph.Kp = static_cast<int32_t>(g.Kp);
    ph.nkb = static_cast<int32_t>(g.Kp / kTileK);
    ph.Nw = static_cast<int32_t>(g.N);
    ph.Nwp = static_cast<int32_t>(g.Np);
    ph.n_tiles = static_cast<int32_t>(g.Np / kTileN);
  }
  prm.padded_offsets = g1.padded_offsets;
  prm.row_to_slot = g1.row_to_slot;
  prm.xs = g1.xs;
  prm.dev_status = g1.dev_status;
  prm.tile_counter = g1.tile_counter;
  prm.e_done = e_done;
  prm.own = own;
  prm.owned = g2.tile_counter;  // the second tile counter: unused by this kernel otherwise
  prm.dbg_hooks = topt.decode_hooks & 3;
  prm.wait_ns = topt.wait_limit_ns;
  prm.withhold = topt.withhold_release;
  prm.hint_ids = hint.ids;
  prm.hint_mask = hint.id_mask;
  prm.hint_off = hint.off;
  prm.hint_slots = hint.slots;
  prm.El = static_cast<int32_t>(g1.El);
  prm.top_k = g1.top_k;
  prm.inter = g1.inter;
  prm.g2 = g1.g2;
  prm.route_w = g2.route_w;
  prm.route_w_dtype = g2.route_w_dtype;
  prm.rsf = g2.rsf;
  const size_t smem = static_cast<size_t>(dgemm::kStages) * dgemm::kStageBytes + dgemm::kSmemExtra +
                      roundup64(g1.El + 1, 4) * 4 + g1.El * 4 + roundup64(g1.El, 16);
  const int64_t units_max = g1.El * (prm.ph[0].n_tiles + prm.ph[1].n_tiles);
  const int grid = static_cast<int>(units_max < num_sms() ? units_max : num_sms());
  prm.n_static = hint.ids != nullptr ? static_cast<int32_t>(grid < kOwnFlags ? grid : kOwnFlags) : 0;
  return dgemm::launch_act(g2.mode == kG2Rows, g1.act, prm, grid, smem, s);
}

}  // namespace moe

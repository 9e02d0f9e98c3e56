// S2: expert-sorted routing plan (moe_sort), a stable counting sort of the routed slots.
//
// Sources: FlashInfer flashinfer.fused_moe.CudnnGroupedGemmNvfp4Config (rows permuted into
// expert order, each expert segment padded to a multiple of 128 rows; non-local experts
// masked; distinct topk_ids per token); Megatron-Core flashinfer_routed_nvfp4_moe (-1
// routing entries contribute zero); FlashInfer flashinfer.fused_moe.FrostLowLatencyConfig
// (expert ids outside [0, num_experts) mark unrouted slots).
// The sort itself is in plan_device.cuh.
//  - one block (small inputs: one launch): histogram, scan, padding fill and placement;
//  - several blocks (large inputs: three launches): per-block histograms, one scan block
//    that turns them into per-block base rows, then per-block placement.
#include "common.cuh"
#include "host_util.h"
#include "plan_device.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(kPlanThreads) plan_single_kernel(
    const int32_t* __restrict__ ids, int id_mask, int64_t n, int top_k, int off, int El, int64_t cap,
    int32_t* __restrict__ counts,
    int32_t* __restrict__ padded_offsets, int32_t* __restrict__ row_to_slot, int32_t* __restrict__ token_to_row,
    int32_t* dev_status) {
  __shared__ PlanSmem sm;
  zero_tables(sm, El);
  pdl_wait();
  pdl_trigger();  // after the wait: a dependent that starts early finds every earlier kernel done
  __syncthreads();
  for (int64_t s = threadIdx.x; s < n; s += blockDim.x) {
    const int l = local_of(entry_id(ids, s, id_mask), off, El);
    if (l >= 0) atomicAdd(&sm.cnt[l], 1);
  }
  __syncthreads();
  scan_padded(sm, El);
  __syncthreads();
  for (int l = threadIdx.x; l <= El; l += blockDim.x) {
    padded_offsets[l] = sm.cursor[l];
    if (l < El) counts[l] = sm.cnt[l];
  }
  fill_padding(sm.cursor, sm.cnt, El, sm.cursor[El], cap, row_to_slot);
  __syncthreads();
  place_range(ids, id_mask, 0, n, top_k, off, El, sm, row_to_slot, token_to_row, dev_status);
}

// per-block histograms: hist[b * El + l]
__global__ void __launch_bounds__(kPlanThreads) plan_hist_kernel(const int32_t* __restrict__ ids, int id_mask,
                                                                 int64_t n, int off, int El,
                                                                 int32_t* __restrict__ hist) {
  __shared__ int cnt[kMaxLocalExperts];
  for (int i = threadIdx.x; i < El; i += blockDim.x) cnt[i] = 0;
  pdl_wait();
  pdl_trigger();  // after the wait: a dependent that starts early finds every earlier kernel done
  __syncthreads();
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kSlotsPerBlock;
  const int64_t b1 = min(n, b0 + kSlotsPerBlock);
  for (int64_t s = b0 + threadIdx.x; s < b1; s += blockDim.x) {
    const int l = local_of(entry_id(ids, s, id_mask), off, El);
    if (l >= 0) atomicAdd(&cnt[l], 1);
  }
  __syncthreads();
  for (int l = threadIdx.x; l < El; l += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * El + l] = cnt[l];
}

// one block: counts, padded offsets, per-block base rows (in place over hist), padding fill
__global__ void __launch_bounds__(kPlanThreads) plan_scan_kernel(int32_t* __restrict__ hist, int nb, int El,
                                                                 int64_t cap, int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ padded_offsets,
                                                                 int32_t* __restrict__ row_to_slot) {
  __shared__ PlanSmem sm;
  constexpr int kBatch = 8;  // independent histogram loads in flight per thread
  pdl_trigger();
  pdl_wait();
  for (int l = threadIdx.x; l < El; l += blockDim.x) {
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += kBatch) {
      int h[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) h[i] = b0 + i < nb ? hist[static_cast<int64_t>(b0 + i) * El + l] : 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) run += h[i];
    }
    sm.cnt[l] = run;
  }
  __syncthreads();
  scan_padded(sm, El);
  __syncthreads();
  // each block's first row per expert, in place over its histogram
  for (int l = threadIdx.x; l <= El; l += blockDim.x) {
    padded_offsets[l] = sm.cursor[l];
    if (l < El) {
      counts[l] = sm.cnt[l];
      int run = sm.cursor[l];
      for (int b0 = 0; b0 < nb; b0 += kBatch) {
        int h[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) h[i] = b0 + i < nb ? hist[static_cast<int64_t>(b0 + i) * El + l] : 0;
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          if (b0 + i < nb) {
            hist[static_cast<int64_t>(b0 + i) * El + l] = run;
            run += h[i];
          }
      }
    }
  }
  fill_padding(sm.cursor, sm.cnt, El, sm.cursor[El], cap, row_to_slot);
}

__global__ void __launch_bounds__(kPlanThreads) plan_place_kernel(const int32_t* __restrict__ ids, int id_mask,
                                                                  int64_t n,
                                                                  int top_k, int off, int El,
                                                                  const int32_t* __restrict__ base,
                                                                  int32_t* __restrict__ row_to_slot,
                                                                  int32_t* __restrict__ token_to_row,
                                                                  int32_t* dev_status) {
  __shared__ PlanSmem sm;
  pdl_trigger();
  zero_warp_counts(sm);
  pdl_wait();
  for (int l = threadIdx.x; l < El; l += blockDim.x) sm.cursor[l] = base[static_cast<int64_t>(blockIdx.x) * El + l];
  __syncthreads();
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kSlotsPerBlock;
  const int64_t b1 = min(n, b0 + kSlotsPerBlock);
  place_range(ids, id_mask, b0, b1, top_k, off, El, sm, row_to_slot, token_to_row, dev_status);
}

int64_t plan_blocks(int64_t n) { return (n + kSlotsPerBlock - 1) / kSlotsPerBlock; }

int id_mask_of(int32_t fmt) { return fmt == MOE_IDS_PACKED ? 0xFFFF : -1; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_plan_capacity(int32_t M, int32_t top_k, int32_t num_local_experts) {
  if (M < 0 || top_k <= 0 || num_local_experts <= 0) return 0;
  const int64_t slots = static_cast<int64_t>(M) * top_k;
  const int64_t segs = slots < num_local_experts ? slots : num_local_experts;
  return static_cast<size_t>(roundup64(slots + (kSegAlign - 1) * segs, kSegAlign));
}

extern "C" size_t moe_plan_workspace_bytes(int32_t M, int32_t top_k, int32_t num_local_experts) {
  if (M < 0 || top_k <= 0 || num_local_experts <= 0) return 0;
  const int64_t n = static_cast<int64_t>(M) * top_k;
  const int64_t nb = plan_blocks(n);
  if (nb <= 1) return 0;
  return static_cast<size_t>(roundup64(nb * num_local_experts * 4, 256));
}

extern "C" moe_status_t moe_plan(const int32_t* topk_ids, int32_t topk_ids_format, int32_t M, int32_t top_k,
                                 int32_t num_experts,
                                 int32_t local_expert_offset, int32_t num_local_experts, int32_t* counts,
                                 int32_t* padded_offsets, int32_t* row_to_slot, int32_t* token_to_row,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
  MOE_CHECK(M >= 0 && top_k >= 1 && num_local_experts >= 1 && num_experts >= 1, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(topk_ids_format == MOE_IDS_INT32 || topk_ids_format == MOE_IDS_PACKED, MOE_ERR_INVALID_ARGUMENT);
  const int id_mask = id_mask_of(topk_ids_format);
  MOE_CHECK(local_expert_offset >= 0 && local_expert_offset + num_local_experts <= num_experts,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(num_local_experts <= kMaxLocalExperts, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(static_cast<int64_t>(M) * top_k < (int64_t(1) << 30), MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(counts && padded_offsets && dev_status, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(counts) && aligned16(padded_offsets) && aligned16(dev_status), MOE_ERR_MISALIGNED);
  const int64_t n = static_cast<int64_t>(M) * top_k;
  const int64_t cap = static_cast<int64_t>(moe_plan_capacity(M, top_k, num_local_experts));
  if (n > 0) {
    MOE_CHECK(topk_ids && row_to_slot && token_to_row, MOE_ERR_INVALID_ARGUMENT);
    MOE_CHECK(aligned16(topk_ids) && aligned16(row_to_slot) && aligned16(token_to_row), MOE_ERR_MISALIGNED);
  }
  const size_t need = moe_plan_workspace_bytes(M, top_k, num_local_experts);
  MOE_CHECK(workspace_bytes >= need, MOE_ERR_WORKSPACE_TOO_SMALL);
  if (need) {
    MOE_CHECK(workspace != nullptr, MOE_ERR_INVALID_ARGUMENT);
    MOE_CHECK(aligned16(workspace), MOE_ERR_MISALIGNED);
  }
  cudaStream_t s = as_stream(stream);
  const int64_t nb = plan_blocks(n);
  const int off = local_expert_offset, El = num_local_experts;
  const dim3 block(kPlanThreads);
  if (nb <= 1)
    return launch_pdl(plan_single_kernel, dim3(1), block, 0, s, topk_ids, id_mask, n, top_k, off, El, cap, counts,
                      padded_offsets, row_to_slot, token_to_row, dev_status);
  int32_t* hist = static_cast<int32_t*>(workspace);
  const dim3 grid(static_cast<unsigned>(nb));
  moe_status_t st = launch_pdl(plan_hist_kernel, grid, block, 0, s, topk_ids, id_mask, n, off, El, hist);
  if (st != MOE_OK) return st;
  st = launch_pdl(plan_scan_kernel, dim3(1), block, 0, s, hist, static_cast<int>(nb), El, cap, counts,
                  padded_offsets, row_to_slot);
  if (st != MOE_OK) return st;
  return launch_pdl(plan_place_kernel, grid, block, 0, s, topk_ids, id_mask, n, top_k, off, El,
                    static_cast<const int32_t*>(hist), row_to_slot, token_to_row, dev_status);
}

// ---------------------------------------------------------------------------------------
// moe_plan_noalloc: the same plan for callers that cannot hand the library device scratch.
//
// Some callers never allocate device memory after start-up: serving runtimes that carve
// all memory from one up-front pool, C hosts without a device allocator of their own, or
// code that must not call cudaMalloc because it would synchronise the device in the middle
// of a stream's work. For them the per-block expert histograms of the multi-block plan
// live in a fixed array in the library's own device memory instead of a workspace.
//
// The array is file-scope device memory, so every GPU that loads the library holds it
// (MOE_PLAN_NOALLOC_SCRATCH_BYTES) until the process exits. In host code its name is only
// a host-side stand-in: the kernels are given the device address that
// cudaGetSymbolAddress returns in the current context. That address is cached per CUDA
// context, keyed by the context's unique id (cuCtxGetId, never reused within a process), so
// a context torn down and re-created (cudaDeviceReset) gets a fresh lookup, never a stale
// address. All calls in a context share the array and it keeps the last call's contents;
// nothing in it has to start at zero (each call writes every histogram entry it later
// reads), but calls that overlap on the GPU (two streams, or two threads) race on it.
// ---------------------------------------------------------------------------------------
#include <mutex>

namespace moe {
namespace {

constexpr int64_t kNoAllocScratchInts = MOE_PLAN_NOALLOC_SCRATCH_BYTES / 4;
static __device__ __align__(256) int32_t g_plan_noalloc_scratch[kNoAllocScratchInts];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(ptr);
}

// unique id of the calling thread's current context, or 0 when it cannot be read
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

constexpr int kCacheSlots = 64;
std::mutex g_noalloc_mu;
unsigned long long g_noalloc_ctx[kCacheSlots] = {};  // context ids (0 = empty slot)
int32_t* g_noalloc_ptr[kCacheSlots] = {};

// device address of the scratch array in the current context (looked up on the first call
// in each context; every call when the context id cannot be read or the cache is full)
moe_status_t noalloc_scratch(int32_t** out) {
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  int free_slot = -1;
  for (int i = 0; id != 0 && i < kCacheSlots; ++i) {
    if (g_noalloc_ctx[i] == id) {
      *out = g_noalloc_ptr[i];
      return MOE_OK;
    }
    if (g_noalloc_ctx[i] == 0 && free_slot < 0) free_slot = i;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_plan_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
  if (id != 0 && free_slot >= 0) {
    g_noalloc_ctx[free_slot] = id;
    g_noalloc_ptr[free_slot] = static_cast<int32_t*>(p);
  }
  *out = static_cast<int32_t*>(p);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_plan_noalloc(const int32_t* topk_ids, int32_t topk_ids_format, int32_t M,
                                         int32_t top_k, int32_t num_experts,
                                         int32_t local_expert_offset, int32_t num_local_experts, int32_t* counts,
                                         int32_t* padded_offsets, int32_t* row_to_slot, int32_t* token_to_row,
                                         int32_t* dev_status, moe_stream_t stream) {
  MOE_CHECK(M >= 0 && top_k >= 1 && num_local_experts >= 1 && num_experts >= 1, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(topk_ids_format == MOE_IDS_INT32 || topk_ids_format == MOE_IDS_PACKED, MOE_ERR_INVALID_ARGUMENT);
  const int id_mask = id_mask_of(topk_ids_format);
  MOE_CHECK(local_expert_offset >= 0 && local_expert_offset + num_local_experts <= num_experts,
            MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(num_local_experts <= kMaxLocalExperts, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(static_cast<int64_t>(M) * top_k < (int64_t(1) << 30), MOE_ERR_UNSUPPORTED_SHAPE);
  const int64_t n = static_cast<int64_t>(M) * top_k;
  const int64_t nb = plan_blocks(n);
  // the histograms must fit the fixed array
  MOE_CHECK(nb <= 1 || nb * num_local_experts <= kNoAllocScratchInts, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK(counts && padded_offsets && dev_status, MOE_ERR_INVALID_ARGUMENT);
  MOE_CHECK(aligned16(counts) && aligned16(padded_offsets) && aligned16(dev_status), MOE_ERR_MISALIGNED);
  if (n > 0) {
    MOE_CHECK(topk_ids && row_to_slot && token_to_row, MOE_ERR_INVALID_ARGUMENT);
    MOE_CHECK(aligned16(topk_ids) && aligned16(row_to_slot) && aligned16(token_to_row), MOE_ERR_MISALIGNED);
  }
  int32_t* hist = nullptr;
  moe_status_t st = noalloc_scratch(&hist);
  if (st != MOE_OK) return st;
  const int64_t cap = static_cast<int64_t>(moe_plan_capacity(M, top_k, num_local_experts));
  cudaStream_t s = as_stream(stream);
  const int off = local_expert_offset, El = num_local_experts;
  if (nb <= 1) {
    plan_single_kernel<<<1, kPlanThreads, 0, s>>>(topk_ids, id_mask, n, top_k, off, El, cap, counts,
                                                  padded_offsets, row_to_slot, token_to_row, dev_status);
    return launch_status();
  }
  plan_hist_kernel<<<static_cast<unsigned>(nb), kPlanThreads, 0, s>>>(topk_ids, id_mask, n, off, El, hist);
  MOE_CHECK(launch_status() == MOE_OK, MOE_ERR_CUDA);
  plan_scan_kernel<<<1, kPlanThreads, 0, s>>>(hist, static_cast<int>(nb), El, cap, counts, padded_offsets,
                                              row_to_slot);
  MOE_CHECK(launch_status() == MOE_OK, MOE_ERR_CUDA);
  plan_place_kernel<<<static_cast<unsigned>(nb), kPlanThreads, 0, s>>>(topk_ids, id_mask, n, top_k, off, El,
                                                                       hist, row_to_slot, token_to_row,
                                                                       dev_status);
  return launch_status();
}

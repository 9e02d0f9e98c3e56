// Device building blocks of the routing plan (moe_sort), shared by the plan kernels and the
// fused small-batch prologue: a stable counting sort of the routed slots into expert
// segments padded to 128 rows.
//
// Slots s = t*top_k + j are placed in ascending s inside each segment. A block places 1024
// slots per step: __match_any_sync groups the lanes of a warp that route to the same
// expert (rank = lower lanes in the group), a 32 x El byte table holds each warp's count
// per expert for the cross-warp prefix, and a per-expert cursor carries the running row.
#pragma once

#include "common.cuh"

namespace moe {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kSlotsPerBlock = 2048;

struct PlanSmem {
  int cnt[kMaxLocalExperts];
  int cursor[kMaxLocalExperts + 1];
  alignas(16) uint8_t warp_cnt[32][kMaxLocalExperts];
};

// the id of a routing entry: all 32 bits (plain ids) or bits 15..0 (packed slots, id_mask 0xFFFF)
__device__ __forceinline__ int entry_id(const int32_t* ids, int64_t s, int id_mask) { return ids[s] & id_mask; }

__device__ __forceinline__ int local_of(int id, int off, int El) {
  const int l = id - off;
  return (l >= 0 && l < El) ? l : -1;
}

// exclusive scan of roundup(cnt[l], 128) by warp 0 into cursor[0..El] (cursor[El] = total)
__device__ void scan_padded(PlanSmem& sm, int El) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int per = (El + 31) / 32;
  int sum = 0;
  for (int i = 0; i < per; ++i) {
    const int l = lane * per + i;
    if (l < El) sum += (sm.cnt[l] + kSegAlign - 1) / kSegAlign * kSegAlign;
  }
  int incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += n;
  }
  int run = incl - sum;
  for (int i = 0; i < per; ++i) {
    const int l = lane * per + i;
    if (l < El) {
      sm.cursor[l] = run;
      run += (sm.cnt[l] + kSegAlign - 1) / kSegAlign * kSegAlign;
    }
  }
  if (lane == 31) sm.cursor[El] = incl;
}

// row_to_slot = -1 on the padding rows of every segment (one warp per expert, lanes across
// its padding rows) and on [total, capacity)
__device__ void fill_padding(const int* start, const int* cnt, int El, int total, int64_t cap,
                             int32_t* row_to_slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int l = warp; l < El; l += nwarps) {
    const int b = start[l] + cnt[l];
    const int e = start[l] + (cnt[l] + kSegAlign - 1) / kSegAlign * kSegAlign;
    for (int p = b + lane; p < e; p += 32) row_to_slot[p] = -1;
  }
  for (int64_t p = total + threadIdx.x; p < cap; p += blockDim.x) row_to_slot[p] = -1;
}

// place slots [begin, end) in order; sm.cursor[l] holds the first free row of expert l.
// row_to_slot and dev_status may be null (a block that only needs token_to_row, which may
// then point to shared memory): the rows are the same, nothing else is written or checked.
__device__ void place_range(const int32_t* __restrict__ ids, int id_mask, int64_t begin, int64_t end, int top_k,
                            int off, int El, PlanSmem& sm, int32_t* __restrict__ row_to_slot, int32_t* __restrict__ token_to_row,
                            int32_t* dev_status) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int64_t base = begin; base < end; base += kPlanThreads) {
    const int64_t s = base + tid;
    int l = -1;
    if (s < end) {
      const int id = entry_id(ids, s, id_mask);
      l = local_of(id, off, El);
      if (l >= 0 && dev_status != nullptr) {
        const int64_t t0 = s - s % top_k;
        for (int64_t q = t0; q < s; ++q)
          if (entry_id(ids, q, id_mask) == id) atomicOr(dev_status, MOE_DEV_DUPLICATE_EXPERT);
      } else if (l < 0) {
        token_to_row[s] = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, l);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = l >= 0 && rank == 0;
    if (leader) sm.warp_cnt[w][l] = static_cast<uint8_t>(__popc(peers));
    __syncthreads();
    if (l >= 0) {
      int prefix = 0;
      for (int ww = 0; ww < w; ++ww) prefix += sm.warp_cnt[ww][l];
      const int row = sm.cursor[l] + prefix + rank;
      if (row_to_slot != nullptr) row_to_slot[row] = static_cast<int32_t>(s);
      token_to_row[s] = row;
    }
    __syncthreads();
    if (leader) {
      atomicAdd(&sm.cursor[l], __popc(peers));
      sm.warp_cnt[w][l] = 0;
    }
    __syncthreads();
  }
}

__device__ void zero_warp_counts(PlanSmem& sm) {
  uint4* w = reinterpret_cast<uint4*>(&sm.warp_cnt[0][0]);
  for (int i = threadIdx.x; i < 32 * kMaxLocalExperts / 16; i += blockDim.x) w[i] = make_uint4(0, 0, 0, 0);
}

__device__ void zero_tables(PlanSmem& sm, int El) {
  for (int i = threadIdx.x; i < El; i += blockDim.x) sm.cnt[i] = 0;
  zero_warp_counts(sm);
}

}  // namespace
}  // namespace moe

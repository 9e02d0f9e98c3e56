// Host-side helpers shared by the C-ABI entry points: argument checks and launch errors.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe_nvfp4.h"

namespace moe {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// [a, a + na) and [b, b + nb) overlap (byte ranges; empty ranges never overlap)
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

inline moe_status_t launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

#define MOE_CHECK(cond, code) \
  do {                        \
    if (!(cond)) return (code); \
  } while (0)

#define MOE_CUDA(call)                                 \
  do {                                                 \
    if ((call) != cudaSuccess) return MOE_ERR_CUDA;    \
  } while (0)

inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// Launch `kern` on `s` with programmatic stream serialisation, so it may begin while the
// previous kernel of the stream finishes (it waits with griddepcontrol.wait before using
// that kernel's results).
template <typename... KArgs, typename... Args>
moe_status_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

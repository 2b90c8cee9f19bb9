// Host-side launch of one kernel instance with programmatic dependent launch
// (shared by the per-head_dim translation units).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "pa_internal.h"

namespace pa {

// Launch `kern(params)` on `grid` CTAs of `threads` threads with `smem` bytes
// of dynamic shared memory, allowing programmatic dependent launch after the
// previous kernel in the stream.  The shared-memory limit is raised once per
// device; `configured` is the instance's own bit set of configured devices.
template <typename Kernel, typename Params>
cudaError_t launch_pdl(Kernel kern, int smem, std::atomic<unsigned long long>& configured,
                       const Params& params, int grid, int threads, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, params);
}

// A split-decode kernel: CTAs of kWarpsPerCta warps.
template <typename Kernel, typename Params>
cudaError_t launch_split_kernel(Kernel kern, int smem, std::atomic<unsigned long long>& configured,
                                const Params& p, int grid, cudaStream_t stream) {
  return launch_pdl(kern, smem, configured, p, grid, kWarpsPerCta * 32, stream);
}

}  // namespace pa

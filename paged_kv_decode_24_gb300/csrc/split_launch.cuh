// Host-side launch of one split-decode kernel instance (shared by the
// per-head_dim translation units).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "decode_kernel.cuh"
#include "pa_internal.h"

namespace pa {

// Launch `kern` on `grid` CTAs of kWarpsPerCta warps with `smem` bytes of
// dynamic shared memory, allowing programmatic dependent launch after the
// previous kernel in the stream.  The shared-memory limit is raised once per
// device; `configured` is the instance's own bit set of configured devices.
template <typename Kernel>
cudaError_t launch_split_kernel(Kernel kern, int smem, std::atomic<unsigned long long>& configured,
                                const SplitParams& p, int grid, cudaStream_t stream) {
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
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace pa

// CUDA-core split-decode kernel for head_dim 64, MHA (G = 1).
#include <atomic>

#include "decode_kernel.cuh"
#include "launch.h"

namespace pa {

namespace {

template <int G>
cudaError_t launch_g(const SplitParams& p, int grid, cudaStream_t stream) {
  constexpr int D = 64;
  constexpr int NSH = half_stages_for(D);
  constexpr int smem = kWarpsPerCta * warp_smem(D, G, NSH).bytes;
  static_assert(smem <= kMaxCtaSmem, "split-decode CTA does not fit in shared memory");
  auto kern = split_decode_kernel<D, G, kWarpsPerCta, NSH>;
  static std::atomic<unsigned long long> configured{0};
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

}  // namespace

cudaError_t launch_split_d64(const SplitParams& p, int group, int grid, cudaStream_t stream) {
  return group == 1 ? launch_g<1>(p, grid, stream) : cudaErrorInvalidValue;
}

}  // namespace pa

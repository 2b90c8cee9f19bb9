// tcgen05 multi-token attention kernel for head_dim 128 (G = 1, 2, 4, 8), fp16 and bf16.
#include "launch.h"
#include "prefill_tc5.cuh"
#include "split_launch.cuh"

namespace pa {

namespace {

template <typename T, int G>
cudaError_t launch_g(const PrefillParams& p, cudaStream_t stream) {
  constexpr int D = 128;
  constexpr int smem = Tc5Layout<D>::BYTES;
  static_assert(smem <= kMaxCtaSmem, "prefill CTA does not fit in shared memory");
  static std::atomic<unsigned long long> configured{0};
  auto kern = prefill_tc5_kernel<T, D, G>;
  return launch_pdl(kern, smem, configured, p, p.num_tiles, kTc5Threads, stream);
}

template <typename T>
cudaError_t launch_t(const PrefillParams& p, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_g<T, 1>(p, stream);
    case 2: return launch_g<T, 2>(p, stream);
    case 4: return launch_g<T, 4>(p, stream);
    case 8: return launch_g<T, 8>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill_tc5_d128(const PrefillParams& p, int group, int dtype,
                                   cudaStream_t stream) {
  if (dtype == PA_DTYPE_BF16) return launch_t<__nv_bfloat16>(p, group, stream);
  return launch_t<__half>(p, group, stream);
}

}  // namespace pa

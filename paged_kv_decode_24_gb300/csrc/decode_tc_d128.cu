// Tensor-core split-decode kernel for head_dim 128, GQA (G = 2, 4, 8), fp16 and bf16.
#include "decode_tc.cuh"
#include "launch.h"
#include "split_launch.cuh"

namespace pa {

namespace {

template <typename T, int G, bool E>
cudaError_t launch_ge(const SplitParams& p, int grid, cudaStream_t stream) {
  constexpr int D = 128;
  constexpr int NSH = half_stages_for(D);
  constexpr int smem = TcLayout<D, kWarpsPerCta, NSH>::BYTES;
  static_assert(smem <= kMaxCtaSmem, "split-decode CTA does not fit in shared memory");
  static std::atomic<unsigned long long> configured{0};
  auto kern = split_decode_tc_kernel<T, D, G, kWarpsPerCta, NSH, E>;
  return launch_split_kernel(kern, smem, configured, p, grid, stream);
}

// The instance of the plan's early_kv: first page copies before (E) or
// after the wait on the previous kernel.
template <typename T, int G>
cudaError_t launch_g(const SplitParams& p, int grid, cudaStream_t stream) {
  return p.early_kv ? launch_ge<T, G, true>(p, grid, stream)
                    : launch_ge<T, G, false>(p, grid, stream);
}

template <typename T>
cudaError_t launch_t(const SplitParams& p, int group, int grid, cudaStream_t stream) {
  switch (group) {
    case 2: return launch_g<T, 2>(p, grid, stream);
    case 4: return launch_g<T, 4>(p, grid, stream);
    case 8: return launch_g<T, 8>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_split_tc_d128(const SplitParams& p, int group, int dtype, int grid, cudaStream_t stream) {
  if (dtype == PA_DTYPE_BF16) return launch_t<__nv_bfloat16>(p, group, grid, stream);
  return launch_t<__half>(p, group, grid, stream);
}

}  // namespace pa

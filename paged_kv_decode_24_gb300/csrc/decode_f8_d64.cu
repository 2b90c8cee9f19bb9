// FP8 (E4M3) cache split-decode kernel for head_dim 64 (G = 1, 2, 4, 8).
#include "decode_q8.cuh"
#include "launch.h"
#include "split_launch.cuh"

namespace pa {

namespace {

template <int G, bool E>
cudaError_t launch_ge(const SplitParams& p, int grid, cudaStream_t stream) {
  constexpr int D = 64;
  constexpr int NS = q8_page_stages_for(D);
  constexpr int smem = Q8Layout<D, kWarpsPerCta, NS>::BYTES;
  static_assert(smem <= kMaxCtaSmem, "split-decode CTA does not fit in shared memory");
  static std::atomic<unsigned long long> configured{0};
  auto kern = split_decode_q8_kernel<D, G, kWarpsPerCta, NS, kCodeE4m3, E>;
  return launch_split_kernel(kern, smem, configured, p, grid, stream);
}

// The instance of the plan's early_kv: first page copies before (E) or
// after the wait on the previous kernel.
template <int G>
cudaError_t launch_g(const SplitParams& p, int grid, cudaStream_t stream) {
  return p.early_kv ? launch_ge<G, true>(p, grid, stream)
                    : launch_ge<G, false>(p, grid, stream);
}

}  // namespace

cudaError_t launch_split_f8_d64(const SplitParams& p, int group, int grid, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_g<1>(p, grid, stream);
    case 2: return launch_g<2>(p, grid, stream);
    case 4: return launch_g<4>(p, grid, stream);
    case 8: return launch_g<8>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa

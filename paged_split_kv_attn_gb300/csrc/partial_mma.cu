// partial_mma.cu -- instantiations of the tensor-core (mma.sync bf16) partial kernel.
#include "partial_kernel.cuh"

namespace pskv {

// Calls f.template operator()<Consumer>() for the tensor-core consumer of (kD, group).
template <int kD, bool kFolded, class F>
static cudaError_t mma_by_group(int group, F &&f) {
  switch (group) {
    case 1: return f.template operator()<MmaConsumer<kD, 1, kFolded>>();
    case 2: return f.template operator()<MmaConsumer<kD, 2, kFolded>>();
    case 4: return f.template operator()<MmaConsumer<kD, 4, kFolded>>();
    case 8: return f.template operator()<MmaConsumer<kD, 8, kFolded>>();
    default: return cudaErrorInvalidValue;
  }
}

template <class F>
static cudaError_t mma_dispatch(int head_dim, int group, bool folded, F &&f) {
  if (head_dim == 512) return folded ? mma_by_group<512, true>(group, f) : mma_by_group<512, false>(group, f);
  if (head_dim == 256) return folded ? mma_by_group<256, true>(group, f) : mma_by_group<256, false>(group, f);
  return cudaErrorInvalidValue;
}

cudaError_t launch_partial_mma(const PartialArgs &a, int head_dim, int group, bool folded,
                               dim3 grid, cudaStream_t s) {
  return mma_dispatch(head_dim, group, folded,
                      [&]<class C>() { return launch_partial_kernel<C>(a, grid, s); });
}

cudaError_t occupancy_partial_mma(int head_dim, int group, bool folded, int *ctas) {
  return mma_dispatch(head_dim, group, folded,
                      [&]<class C>() { return partial_kernel_occupancy<C>(ctas); });
}

}  // namespace pskv

// partial_mma.cu -- instantiations of the tensor-core (mma.sync bf16) partial kernel.
#include "partial_kernel.cuh"

namespace pskv {

// Calls f.template operator()<Consumer>() for the tensor-core consumer of (kD, group).
template <int kD, class F>
static cudaError_t mma_by_group(int group, F &&f) {
  switch (group) {
    case 1: return f.template operator()<MmaConsumer<kD, 1>>();
    case 2: return f.template operator()<MmaConsumer<kD, 2>>();
    case 4: return f.template operator()<MmaConsumer<kD, 4>>();
    case 8: return f.template operator()<MmaConsumer<kD, 8>>();
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_partial_mma(const PartialArgs &a, int head_dim, int group, dim3 grid,
                               cudaStream_t s) {
  auto launch = [&]<class C>() { return launch_partial_kernel<C>(a, grid, s); };
  if (head_dim == 512) return mma_by_group<512>(group, launch);
  if (head_dim == 256) return mma_by_group<256>(group, launch);
  return cudaErrorInvalidValue;
}

cudaError_t occupancy_partial_mma(int head_dim, int group, int *ctas) {
  auto query = [&]<class C>() { return partial_kernel_occupancy<C>(ctas); };
  if (head_dim == 512) return mma_by_group<512>(group, query);
  if (head_dim == 256) return mma_by_group<256>(group, query);
  return cudaErrorInvalidValue;
}

}  // namespace pskv

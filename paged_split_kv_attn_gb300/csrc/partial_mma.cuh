// partial_mma.cuh -- dispatch of the tensor-core (mma.sync bf16) partial kernel
// over (head dim, group, format) for one count of query n-tiles.
#pragma once
#include "partial_kernel.cuh"

namespace pskv {

// Calls f.template operator()<Consumer>() for the tensor-core consumer of (kD, group).
template <int kD, bool kFolded, int kNT, bool kTree, class F>
static cudaError_t mma_by_group(int group, F &&f) {
  switch (group) {
    case 1: return f.template operator()<MmaConsumer<kD, 1, kFolded, kNT, kTree>>();
    case 2: return f.template operator()<MmaConsumer<kD, 2, kFolded, kNT, kTree>>();
    case 4: return f.template operator()<MmaConsumer<kD, 4, kFolded, kNT, kTree>>();
    case 8: return f.template operator()<MmaConsumer<kD, 8, kFolded, kNT, kTree>>();
    default: return cudaErrorInvalidValue;
  }
}

template <int kNT, bool kTree, class F>
static cudaError_t mma_dispatch(int head_dim, int group, bool folded, F &&f) {
  if (head_dim == 512)
    return folded ? mma_by_group<512, true, kNT, kTree>(group, f)
                  : mma_by_group<512, false, kNT, kTree>(group, f);
  if (head_dim == 256)
    return folded ? mma_by_group<256, true, kNT, kTree>(group, f)
                  : mma_by_group<256, false, kNT, kTree>(group, f);
  return cudaErrorInvalidValue;
}

template <int kNT, bool kTree>
cudaError_t launch_partial_mma_nt(const PartialArgs &a, int head_dim, int group, bool folded,
                                  dim3 grid, cudaStream_t s) {
  return mma_dispatch<kNT, kTree>(head_dim, group, folded,
                                  [&]<class C>() { return launch_partial_kernel<C>(a, grid, s); });
}

template <int kNT>
cudaError_t occupancy_partial_mma_nt(int head_dim, int group, bool folded, int *ctas) {
  return mma_dispatch<kNT, false>(head_dim, group, folded,
                                  [&]<class C>() { return partial_kernel_occupancy<C>(ctas); });
}

// One translation unit instantiates each n-tile count, and one the drafted-tree
// kernels of both counts (compiled in parallel).
extern template cudaError_t launch_partial_mma_nt<1, false>(const PartialArgs &, int, int, bool,
                                                            dim3, cudaStream_t);
extern template cudaError_t launch_partial_mma_nt<2, false>(const PartialArgs &, int, int, bool,
                                                            dim3, cudaStream_t);
extern template cudaError_t launch_partial_mma_nt<1, true>(const PartialArgs &, int, int, bool,
                                                           dim3, cudaStream_t);
extern template cudaError_t launch_partial_mma_nt<2, true>(const PartialArgs &, int, int, bool,
                                                           dim3, cudaStream_t);
extern template cudaError_t occupancy_partial_mma_nt<1>(int, int, bool, int *);
extern template cudaError_t occupancy_partial_mma_nt<2>(int, int, bool, int *);

}  // namespace pskv

// partial_mma.cu -- the tensor-core partial kernel with one n-tile of query
// columns (single-token decode and short verify windows), and the dispatch on
// the n-tile count.
#include "partial_mma.cuh"

namespace pskv {

template cudaError_t launch_partial_mma_nt<1, false>(const PartialArgs &, int, int, bool, dim3,
                                                     cudaStream_t);
template cudaError_t occupancy_partial_mma_nt<1>(int, int, bool, int *);

cudaError_t launch_partial_mma(const PartialArgs &a, int head_dim, int group, bool folded, int nt,
                               dim3 grid, cudaStream_t s) {
  const bool tree = a.tree_mask != nullptr;
  if (nt == 1)
    return tree ? launch_partial_mma_nt<1, true>(a, head_dim, group, folded, grid, s)
                : launch_partial_mma_nt<1, false>(a, head_dim, group, folded, grid, s);
  if (nt == 2)
    return tree ? launch_partial_mma_nt<2, true>(a, head_dim, group, folded, grid, s)
                : launch_partial_mma_nt<2, false>(a, head_dim, group, folded, grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t occupancy_partial_mma(int head_dim, int group, bool folded, int nt, int *ctas) {
  if (nt == 1) return occupancy_partial_mma_nt<1>(head_dim, group, folded, ctas);
  if (nt == 2) return occupancy_partial_mma_nt<2>(head_dim, group, folded, ctas);
  return cudaErrorInvalidValue;
}

}  // namespace pskv

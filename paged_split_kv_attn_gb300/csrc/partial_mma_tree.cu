// partial_mma_tree.cu -- the tensor-core partial kernel for drafted trees
// (window keys visible by each token's ancestor mask), with one and two
// n-tiles of query columns.
#include "partial_mma.cuh"

namespace pskv {

template cudaError_t launch_partial_mma_nt<1, true>(const PartialArgs &, int, int, bool, dim3,
                                                    cudaStream_t);
template cudaError_t launch_partial_mma_nt<2, true>(const PartialArgs &, int, int, bool, dim3,
                                                    cudaStream_t);

}  // namespace pskv

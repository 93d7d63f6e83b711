// partial_mma_nt2.cu -- the tensor-core partial kernel with two n-tiles of
// query columns (verify windows of 9 to 16 query columns per KV head).
#include "partial_mma.cuh"

namespace pskv {

template cudaError_t launch_partial_mma_nt<2, false>(const PartialArgs &, int, int, bool, dim3,
                                                     cudaStream_t);
template cudaError_t occupancy_partial_mma_nt<2>(int, int, bool, int *);

}  // namespace pskv

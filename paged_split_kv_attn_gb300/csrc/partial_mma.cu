// partial_mma.cu -- instantiations of the tensor-core (mma.sync bf16) partial kernel.
#include "partial_kernel.cuh"

namespace pskv {

cudaError_t launch_partial_mma(const PartialArgs &a, int head_dim, dim3 grid, cudaStream_t s) {
  if (head_dim == 512) return launch_partial_kernel<MmaConsumer<512>>(a, grid, s);
  if (head_dim == 256) return launch_partial_kernel<MmaConsumer<256>>(a, grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t occupancy_partial_mma(int head_dim, int *ctas) {
  if (head_dim == 512) return partial_kernel_occupancy<MmaConsumer<512>>(ctas);
  if (head_dim == 256) return partial_kernel_occupancy<MmaConsumer<256>>(ctas);
  return cudaErrorInvalidValue;
}

}  // namespace pskv

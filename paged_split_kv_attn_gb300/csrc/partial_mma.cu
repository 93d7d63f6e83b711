// partial_mma.cu -- instantiations of the tensor-core (mma.sync bf16) partial kernel.
#include "partial_kernel.cuh"

namespace pskv {

cudaError_t launch_partial_mma(const PartialArgs &a, int head_dim, dim3 grid, cudaStream_t s) {
  if (head_dim == 512) return launch_partial_kernel<MmaConsumer<512>>(a, grid, s);
  if (head_dim == 256) return launch_partial_kernel<MmaConsumer<256>>(a, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace pskv

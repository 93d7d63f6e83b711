// partial_simt_f32.cu -- instantiations of the CUDA-core partial kernel for f32 pools.
#include "partial_kernel.cuh"

namespace pskv {

template <int kD>
static cudaError_t by_group(const PartialArgs &a, int group, dim3 grid, cudaStream_t s) {
  switch (group) {
    case 1: return launch_partial_kernel<SimtConsumer<float, kD, 1>>(a, grid, s);
    case 2: return launch_partial_kernel<SimtConsumer<float, kD, 2>>(a, grid, s);
    case 4: return launch_partial_kernel<SimtConsumer<float, kD, 4>>(a, grid, s);
    case 8: return launch_partial_kernel<SimtConsumer<float, kD, 8>>(a, grid, s);
    default: break;
  }
  if constexpr (kD == 256) {
    if (group == 16) return launch_partial_kernel<SimtConsumer<float, kD, 16>>(a, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_partial_simt_f32(const PartialArgs &a, int head_dim, int group, dim3 grid,
                                    cudaStream_t s) {
  if (head_dim == 512) return by_group<512>(a, group, grid, s);
  if (head_dim == 256) return by_group<256>(a, group, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace pskv

// Sliced-key backward with the chunk count as a template constant (rows up
// to 2560 wide), instantiated for the f32 storage dtype.
#include "kernels_lr.cuh"

namespace ar {
template cudaError_t dispatch_lr_bwd_fixed<float>(const RouteArgs *a, cudaStream_t s, int *grid_warps);
}  // namespace ar

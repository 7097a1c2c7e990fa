// Backward routing kernels instantiated for the f32 storage dtype.
#include "kernels_bwd.cuh"

namespace ar {
template cudaError_t dispatch_bwd<float>(const RouteArgs *a, cudaStream_t s, int *grid_warps);
}  // namespace ar

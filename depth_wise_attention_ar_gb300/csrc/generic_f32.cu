// Scalar-access routing kernels (shapes outside the tiled families)
// instantiated for the fp32 storage dtype.
#include "kernels_generic.cuh"

namespace ar {
template cudaError_t dispatch_generic_fwd<float>(const RouteArgs &a, cudaStream_t s);
template cudaError_t dispatch_coupling<float>(const RouteArgs &a, float *S, cudaStream_t s);
template cudaError_t dispatch_generic_bwd<float>(const RouteArgs *a, cudaStream_t s, int *grid_warps);
}  // namespace ar

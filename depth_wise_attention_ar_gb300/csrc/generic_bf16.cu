// Scalar-access routing kernels (shapes outside the tiled families)
// instantiated for the bf16 storage dtype.
#include "kernels_generic.cuh"

namespace ar {
template cudaError_t dispatch_generic_fwd<__nv_bfloat16>(const RouteArgs &a, cudaStream_t s);
template cudaError_t dispatch_coupling<__nv_bfloat16>(const RouteArgs &a, float *S, cudaStream_t s);
template cudaError_t dispatch_generic_bwd<__nv_bfloat16>(const RouteArgs *a, cudaStream_t s, int *grid_warps);
}  // namespace ar

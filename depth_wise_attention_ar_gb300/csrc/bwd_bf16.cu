// Backward routing kernels instantiated for the bf16 storage dtype.
#include "kernels_bwd.cuh"

namespace ar {
template cudaError_t dispatch_bwd<__nv_bfloat16>(const RouteArgs *a, cudaStream_t s, int *grid_warps);
}  // namespace ar

// Four-warp (wide-row) routing kernels instantiated for the bf16 storage dtype.
#include "kernels_coop.cuh"

namespace ar {
template cudaError_t dispatch_coop_fwd<__nv_bfloat16>(const RouteArgs &a, cudaStream_t s);
template cudaError_t dispatch_coop_bwd<__nv_bfloat16>(const RouteArgs *a, cudaStream_t s, int *grid_rows);
}  // namespace ar

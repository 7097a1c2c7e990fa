// Four-warp (wide-row) routing kernels instantiated for the f32 storage dtype.
#include "kernels_coop.cuh"

namespace ar {
template cudaError_t dispatch_coop_fwd<float>(const RouteArgs &a, cudaStream_t s);
template cudaError_t dispatch_coop_bwd<float>(const RouteArgs *a, cudaStream_t s, int *grid_rows);
}  // namespace ar

// Sliced-key (r < d) routing kernels instantiated for the f32 storage dtype.
#include "kernels_lr.cuh"

namespace ar {
// rows up to 2560 wide: instantiated in lrfix_f32.cu
extern template cudaError_t dispatch_lr_bwd_fixed<float>(const RouteArgs *a, cudaStream_t s,
                                                      int *grid_warps);
template cudaError_t dispatch_lr_fwd<float>(const RouteArgs &a, cudaStream_t s);
template cudaError_t dispatch_lr_bwd<float>(const RouteArgs *a, cudaStream_t s, int *grid_warps);
}  // namespace ar

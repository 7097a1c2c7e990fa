// Sliced-key (r < d) routing kernels instantiated for the bf16 storage dtype.
#include "kernels_lr.cuh"

namespace ar {
// rows up to 2560 wide: instantiated in lrfix_bf16.cu
extern template cudaError_t dispatch_lr_bwd_fixed<__nv_bfloat16>(const RouteArgs *a, cudaStream_t s,
                                                      int *grid_warps);
template cudaError_t dispatch_lr_fwd<__nv_bfloat16>(const RouteArgs &a, cudaStream_t s);
template cudaError_t dispatch_lr_bwd<__nv_bfloat16>(const RouteArgs *a, cudaStream_t s, int *grid_warps);
}  // namespace ar

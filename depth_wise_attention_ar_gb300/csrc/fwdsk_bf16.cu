// Single-pass sliced-key forward instantiated for the bf16 storage dtype.
#include "kernels_fwd.cuh"

namespace ar {
template cudaError_t dispatch_fwd_sk<__nv_bfloat16>(const RouteArgs &a, cudaStream_t s);
}  // namespace ar

// Single-pass sliced-key forward instantiated for the f32 storage dtype.
#include "kernels_fwd.cuh"

namespace ar {
template cudaError_t dispatch_fwd_sk<float>(const RouteArgs &a, cudaStream_t s);
}  // namespace ar

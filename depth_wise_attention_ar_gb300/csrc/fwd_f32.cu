// Forward routing kernels instantiated for the f32 storage dtype.
#include "kernels_fwd.cuh"

namespace ar {
template cudaError_t dispatch_fwd<float>(const RouteArgs &a, cudaStream_t s);
}  // namespace ar

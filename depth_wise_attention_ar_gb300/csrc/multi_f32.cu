// Multi-query forward instantiated for the f32 storage dtype.
#include "kernels_multi.cuh"

namespace ar {
template cudaError_t dispatch_fwd_multi<float>(const MultiArgs &m, cudaStream_t s);
}  // namespace ar

// Multi-query forward instantiated for the bf16 storage dtype.
#include "kernels_multi.cuh"
#include "kernels_multi_mma.cuh"

namespace ar {
template cudaError_t dispatch_fwd_multi<__nv_bfloat16>(const MultiArgs &m, cudaStream_t s);
}  // namespace ar

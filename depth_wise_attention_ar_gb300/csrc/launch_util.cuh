// Launch-configuration cache: dynamic shared-memory opt-in and persistent grid
// size (SM count x resident blocks per SM), computed once per kernel, shared
// memory size and device.
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

namespace ar {

inline cudaError_t persistent_grid(const void *kern, int threads, size_t smem, int *grid)
{
    static std::mutex mu;
    static std::map<std::tuple<const void *, size_t, int>, int> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_tuple(kern, smem, dev);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *grid = it->second;
        return cudaSuccess;
    }
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    *grid = sms * per_sm;
    cache[key] = *grid;
    return cudaSuccess;
}

}  // namespace ar

// Launch-configuration cache: dynamic shared-memory opt-in and persistent grid
// size (SM count x resident blocks per SM), computed once per kernel, shared
// memory size and device.
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

namespace ar {

inline cudaError_t persistent_grid(const void *kern, int threads, size_t smem, int *grid)
{
    static std::mutex mu;
    static std::map<std::tuple<const void *, size_t, int>, int> cache;
    // the dynamic shared-memory opt-in of each kernel only grows: a kernel
    // launched with several sizes keeps the largest, so every cached size fits
    static std::map<std::pair<const void *, int>, size_t> opt_in;
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
    size_t &cap = opt_in[std::make_pair(kern, dev)];
    if (smem > 48 * 1024 && smem > cap) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cap = smem;
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

// ar_route_bwd_noalloc: the routing backward with its scratch in a fixed
// device array owned by this library, for callers that cannot allocate
// device memory themselves.
//
// Who needs it: code that runs under a device-memory budget fixed before it
// starts, with no allocator of its own — for example a plugin whose execute
// hook in a host engine may not call cudaMalloc, or a library embedded in a
// process whose device memory is owned by another framework's pool. Such a
// caller still provides inputs and outputs; only the backward's workspace
// (the per-block dq/dg partial sums) moves into this file's static array.
//
// The array is a file-scope __device__ object: every GPU on which this
// library's device code is loaded holds it (kNoAllocScratchBytes) until the
// process exits. Under CUDA's lazy module loading (the default) the code, and
// with it the array, is loaded on a device when the library is first used
// there, which may be the first call of this entry point (its address lookup):
// a caller with a fixed memory budget should count the array from that first
// call on. Its device address is looked up once per device, on the first call
// made with that device current; make that first call before any stream
// capture. Devices are numbered 0..63 here; a call with a higher device
// current returns AR_ERR_CUDA. The
// address is kept for the life of the process, so a cudaDeviceReset between
// uses (which unloads this code and its array) is not supported. Every call
// shares the one array: calls whose kernels may overlap on the GPU (different
// streams without ordering between them) race on it and must be serialised by
// the caller. Nothing in it has to start at zero: the backward writes every
// partial it later sums, so the previous call's contents are never read.
#include <cuda_runtime.h>

#include <mutex>

#include "attnres.h"
#include "ar_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = AR_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of g_noalloc_scratch, per device (host code must not use the
// symbol itself as a pointer: on the host it is only a stand-in).
void *scratch_for_current_device(ar_status *st)
{
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        *st = AR_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            *st = AR_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    *st = AR_OK;
    return addr[dev];
}

}  // namespace

extern "C" ar_status ar_noalloc_scratch_bytes(size_t *bytes)
{
    if (!bytes) return AR_ERR_INVALID_ARG;
    *bytes = kNoAllocScratchBytes;
    return AR_OK;
}

extern "C" ar_status ar_route_bwd_noalloc(ar_bank *bank, const int32_t *rows, int32_t n_src,
                                          int32_t H, const float *q, const float *g,
                                          const void *out, const void *dout, const float *lse,
                                          float *dq, float *dg, int32_t site_id, void *stream)
{
    if (ar::bank_device_check(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    size_t need = 0;
    ar_status st = ar_route_bwd_workspace(bank, H, &need);
    if (st != AR_OK) return st;
    if (need > kNoAllocScratchBytes) return AR_ERR_CAPACITY;  // beyond the fixed scratch
    void *scratch = scratch_for_current_device(&st);
    if (st != AR_OK) return st;
    return ar_route_bwd(bank, rows, n_src, H, q, g, out, dout, lse, dq, dg, scratch,
                        kNoAllocScratchBytes, site_id, stream);
}

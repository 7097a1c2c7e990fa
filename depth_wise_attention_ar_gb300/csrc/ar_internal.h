// Host-visible internals shared by the C-ABI layer and the kernel units:
// the argument block of a routing launch and the launch entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "attnres.h"

namespace ar {

#ifdef AR_CHECKED
// Range checks of the checked build: the buffers one launch may touch.
// bank and grad are [cap, T, d] row arrays (an access must lie inside one
// row the site lists); every other buffer is a span [lo, hi), writable or not.
constexpr int kCheckSpans = 48;
struct CheckTable {
    uint64_t bank, bank_row, grad, grad_row;  // bases and bytes per row
    int cap;
    int n;
    uint64_t lo[kCheckSpans], hi[kCheckSpans];
    uint8_t wr[kCheckSpans];
    unsigned long long *fault;  // [taken, address, kind << 32 | bytes]
    int off;                    // 1: this launch is not checked
};
#endif

// Everything a routing launch needs, passed by value (kernel parameter space).
struct RouteArgs {
    const void *bank;      // rows [cap, T, d] of the storage dtype
    const float *inv;      // inverse RMS, token-major [T, inv_ld]
    float *grad;           // fp32 gradient rows [cap, T, d] (backward)
    const float *q;        // [r], element stride q_stride
    const float *g;        // [r], element stride g_stride, or nullptr (= ones)
    void *out;             // forward output [T, d]
    float *lse;            // [T, H]
    const void *fout;      // backward: forward output [T, d]
    const void *dout;      // backward: dL/dout [T, d]
    float *ws;             // backward: per-warp partial sums [warps, r]
    unsigned int *err;     // device error word
    // delta form (h = partial + alpha * routed): forward epilogue and backward
    const void *partial;   // forward: residual stream [T, d], or nullptr
    const float *alpha;    // gate (device scalar), or nullptr (= 1)
    void *routed;          // forward: also store the routed mix here, or nullptr
    float *dalpha;         // backward: dL/dalpha (device scalar), or nullptr
    int64_t T;
    int64_t q_stride, g_stride;  // elements between consecutive entries of q, g
    int d, r, H, n_src, inv_ld, norm_full;
    int grad_v8;           // gradient rows' base is 32-byte aligned: 256-bit stores
    // forward with the append fused in: 1 + the list index of the row appended
    // in this call, whose inverse RMS the kernel computes and caches (0: none)
    int fresh1;
    float eps;             // the bank's RMSNorm epsilon
    // the fused append's source when the new row is not already in its slot:
    // new = fresh_src (copy) or row acc_row + fresh_src (block partial sum),
    // written to its slot by the forward; acc_row = -1 for a copy
    const void *fresh_src;
    int acc_row;
    // polls of an mbarrier wait before it is declared lost (0: kWaitLimit);
    // with lost_copies set (a test of the failure path, one-warp full-key
    // forward only) every stage is armed for its bytes but no copy is issued,
    // so the first wait of every warp runs out with nothing in flight
    uint32_t wait_limit;
    int lost_copies;
    int rows[AR_MAX_SOURCES];
    // a row listed k > 1 times in a site enters once with log k added to its
    // score (softmax over the list = softmax over distinct rows with weights k)
    int has_bias;
    float bias[AR_MAX_SOURCES];
    uint32_t first_mask[AR_MAX_SOURCES / 32];  // backward: bit n set = store (first touch)
    // backward: the coupling term S [T, H] summed exactly over the sources
    // (route_coupling_kernel), read instead of <G_h, out_h>; nullptr: from out
    const float *coupling;
#ifdef AR_CHECKED
    CheckTable chk;
#endif
};

// The multi-query forward's arguments: the shared fields plus one query,
// norm weight, output and lse per site.
struct MultiArgs {
    RouteArgs base;
    int nq;
    const float *q[AR_MAX_QUERIES];
    const float *g[AR_MAX_QUERIES];
    void *out[AR_MAX_QUERIES];
    float *lse[AR_MAX_QUERIES];
};

// ---- host-side launch entry points (one per kernel family) -----------------
// Each returns cudaErrorNotSupported when no instantiation covers the shape.
cudaError_t launch_route_fwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s);
cudaError_t launch_route_bwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s);
// The exact coupling term of a site's backward into S [T, H] (fp32).
cudaError_t launch_route_coupling(const RouteArgs &a, float *S, ar_dtype dt, cudaStream_t s);
cudaError_t launch_route_fwd_multi(const MultiArgs &m, ar_dtype dt, cudaStream_t s);
cudaError_t dispatch_fwd_multi_mma(const MultiArgs &m, cudaStream_t s);  // bf16 rows
cudaError_t route_bwd_grid(const RouteArgs &a, ar_dtype dt, int *grid_warps);
// The site runs on a forward kernel that can take the append of a listed row:
// with the row in its slot (in_place) the one-warp full-key kernels on rows up
// to 1024 wide and the four-warp kernels; with a copy or a partial sum to
// form, the four-warp kernels.
bool fwd_fuses_append(const RouteArgs &a, ar_dtype dt, bool in_place);
// dq and dg are written with the strides of q and g respectively.
// The launches below take, last, the buffer table of the range-checked build
// (its chk field; ignored by the normal build, and nullptr = not checked).
cudaError_t launch_dqdg_reduce(const float *ws, int rows, int r, const float *q, int64_t q_stride,
                               const float *g, int64_t g_stride, float *dq, float *dg,
                               float *dalpha, cudaStream_t s, const RouteArgs *chk = nullptr);
cudaError_t launch_merge(const void *oa, const float *la, const void *ob, const float *lb,
                         void *out, float *lse, int64_t T, int d, int H, ar_dtype dt, cudaStream_t s,
                         const RouteArgs *chk = nullptr);
cudaError_t launch_token_sum(const float *grad, int64_t T, int d, float *out, cudaStream_t s,
                             const RouteArgs *chk = nullptr);
// src is a strided [T, d] view: element (t, c) at src[t * ld + c * es]
// (ld = 0: the same vector for every token).
cudaError_t launch_append(const void *src, const void *prev, void *dst, float *inv_col,
                          int64_t T, int d, int r, int inv_ld, int norm_full, float eps,
                          ar_dtype dt, cudaStream_t s, int64_t ld, int64_t es,
                          const RouteArgs *chk = nullptr);
cudaError_t launch_grad_fold(float *dst, const float *src, int64_t n, bool src_valid,
                             bool dst_valid, cudaStream_t s, const RouteArgs *chk = nullptr);
unsigned int *device_error_word();
#ifdef AR_CHECKED
// The checked build's record of the first refused access (three words).
unsigned long long *device_check_fault();
#endif
// AR_OK when the current device is the one the bank was created on (or the
// bank's device is unknown), else AR_ERR_INVALID_ARG: every launch runs on the
// current device, and the bank's buffers belong to its own.
ar_status bank_device_check(const ar_bank *b);
// Some kernel family serves n_src distinct rows at this shape (`repeats`: the
// site lists a row more than once).
bool route_supported(int d, int r, int H, int n_src, ar_dtype dt, bool repeats);
// Workspace rows of the scalar-access backward on the current device; any
// site may run there (repeated rows, or a key cache too large for the
// sliced-key kernels), so every workspace holds at least this many rows.
cudaError_t generic_bwd_rows(int *rows);

// Shapes of the four-warp kernels: d = 1024 * CPL (CPL in 1..8), H a multiple
// of 4 with H/4 heads per warp a power of two <= 32; r = d, or r = k * d/4
// (k in 1..3) with H/k a power of two <= 32.
inline bool coop_supported(int d, int r, int H)
{
    if (d <= 0 || d % 1024 != 0 || d / 1024 > 8) return false;
    if (H < 4 || H % 4 != 0 || H / 4 > 32 || (32 % (H / 4)) != 0) return false;
    if (r == d) return true;
    const int CG = d / 4;
    if (r <= 0 || r % CG != 0 || r > d) return false;
    const int kw = r / CG;
    return H % kw == 0 && H / kw <= 32 && (32 % (H / kw)) == 0;
}

}  // namespace ar

// Bank append (+ inverse RMS), the fixed-order dq/dg reduction, the device
// error word, and the dtype dispatch of the routing launches.
#include "common.cuh"
#include "launch_util.cuh"

namespace ar {

template <typename T> cudaError_t dispatch_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps);
template <typename T> cudaError_t dispatch_lr_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_lr_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps);

// Device error word; kernels get its address as an argument.
__device__ unsigned int g_device_error = 0;

unsigned int *device_error_word()
{
    // cached per device: the symbol lookup is done once, outside any capture
    static unsigned int *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int *>(p);
    }
    return cache[dev];
}

// ---- append ----------------------------------------------------------------
// One warp per token. new = src (copied only when src is not the slot
// itself), or prev + src in fp32 rounded once to the storage dtype (block
// partial sums, "Low-Rank Attention Residuals" Sec. 3.3 / Figure 11). The
// inverse RMS is taken over the stored (rounded) values of the RMS
// coordinates: the last r ("Low-Rank Attention Residuals" Eq. 11/13), or all
// d for the full-width norm ("Multi-Head Attention Residuals" Appendix E).
template <typename T>
__global__ void __launch_bounds__(256) append_kernel(const T *src, const T *prev, T *dst, float *inv,
                                                     int64_t TT, int d, int r, int inv_ld,
                                                     int norm_full, float eps)
{
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nch = d / 8;
    const int c0 = norm_full ? 0 : (d - r) / 8;
    const float inv_w = 1.0f / (float)(norm_full ? d : r);
    const bool write = (src != dst) || prev != nullptr;
    for (int64_t t = w0; t < TT; t += nw) {
        const T *s = src + t * d;
        T *o = dst + t * d;
        float ss = 0.f;
        if (write) {
            for (int c = lane; c < nch; c += 32) {
                float x[8];
                ld_chunk_g(s + c * 8, x);
                if (prev) {
                    float p[8];
                    ld_chunk_g(prev + t * d + c * 8, p);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] += p[e];
                }
                st_chunk_g(o + c * 8, x);
                if (c >= c0) {
                    if constexpr (sizeof(T) == 2) {
                        // square the stored (rounded) value
                        float xr[8];
                        uint4 u;
                        u.x = pack_bf16x2(x[0], x[1]);
                        u.y = pack_bf16x2(x[2], x[3]);
                        u.z = pack_bf16x2(x[4], x[5]);
                        u.w = pack_bf16x2(x[6], x[7]);
                        unpack_bf16x8(u, xr);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(xr[e], xr[e], ss);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
                    }
                }
            }
        } else {
            for (int c = c0 + lane; c < nch; c += 32) {
                float x[8];
                ld_chunk_g(o + c * 8, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) inv[t * inv_ld] = rsqrtf(fmaf(ss, inv_w, eps));
    }
}

cudaError_t launch_append(const void *src, const void *prev, void *dst, float *inv_col, int64_t T,
                          int d, int r, int inv_ld, int norm_full, float eps, ar_dtype dt,
                          cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    int grid = 0;
    const void *k = dt == AR_BF16 ? reinterpret_cast<const void *>(&append_kernel<__nv_bfloat16>)
                                  : reinterpret_cast<const void *>(&append_kernel<float>);
    cudaError_t e = persistent_grid(k, 256, 0, &grid);
    if (e != cudaSuccess) return e;
    const int64_t need = (T + 7) / 8;
    if (need < grid) grid = (int)need;
    if (dt == AR_BF16)
        append_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(src), static_cast<const __nv_bfloat16 *>(prev),
            static_cast<__nv_bfloat16 *>(dst), inv_col, T, d, r, inv_ld, norm_full, eps);
    else
        append_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(src),
                                                  static_cast<const float *>(prev),
                                                  static_cast<float *>(dst), inv_col, T, d, r,
                                                  inv_ld, norm_full, eps);
    return cudaGetLastError();
}

// ---- dq / dg -----------------------------------------------------------------
// dq_c = g_c * sum_w ws[w, c], dg_c = q_c * sum_w ws[w, c]; the sum over the
// backward's warps runs in a fixed order (8 strided groups, then the groups
// in order), so repeated runs give identical bits.
__global__ void __launch_bounds__(256) dqdg_reduce_kernel(const float *ws, int rows, int r,
                                                          const float *q, const float *g,
                                                          float *dq, float *dg)
{
    __shared__ float part[8][33];
    const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (c < r)
        for (int w = grp; w < rows; w += 8) s += ws[(int64_t)w * r + c];
    part[grp][lane] = s;
    __syncthreads();
    if (grp == 0 && c < r) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) t += part[k][lane];
        dq[c] = (g ? g[c] : 1.0f) * t;
        if (dg) dg[c] = q[c] * t;
    }
}

cudaError_t launch_dqdg_reduce(const float *ws, int rows, int r, const float *q, const float *g,
                               float *dq, float *dg, cudaStream_t s)
{
    dqdg_reduce_kernel<<<(r + 31) / 32, 256, 0, s>>>(ws, rows, r, q, g, dq, dg);
    return cudaGetLastError();
}

// ---- dtype / key-width dispatch ------------------------------------------------
// r = d: full-width keys (online-softmax forward, register-resident state);
// r < d: sliced keys (two-sweep forward with a key cache, blocked backward).
cudaError_t launch_route_fwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s)
{
    if (a.r < a.d)
        return dt == AR_BF16 ? dispatch_lr_fwd<__nv_bfloat16>(a, s) : dispatch_lr_fwd<float>(a, s);
    return dt == AR_BF16 ? dispatch_fwd<__nv_bfloat16>(a, s) : dispatch_fwd<float>(a, s);
}

cudaError_t launch_route_bwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s)
{
    if (a.r < a.d)
        return dt == AR_BF16 ? dispatch_lr_bwd<__nv_bfloat16>(&a, s, nullptr)
                             : dispatch_lr_bwd<float>(&a, s, nullptr);
    return dt == AR_BF16 ? dispatch_bwd<__nv_bfloat16>(&a, s, nullptr)
                         : dispatch_bwd<float>(&a, s, nullptr);
}

cudaError_t route_bwd_grid(const RouteArgs &a, ar_dtype dt, int *grid_warps)
{
    if (a.r < a.d)
        return dt == AR_BF16 ? dispatch_lr_bwd<__nv_bfloat16>(&a, nullptr, grid_warps)
                             : dispatch_lr_bwd<float>(&a, nullptr, grid_warps);
    return dt == AR_BF16 ? dispatch_bwd<__nv_bfloat16>(&a, nullptr, grid_warps)
                         : dispatch_bwd<float>(&a, nullptr, grid_warps);
}

bool fused_shape_supported(int d, int r, int H)
{
    if (H < 1 || H > 32 || (32 % H) != 0) return false;
    if (d <= 0 || r <= 0 || r > d || d % 256 != 0 || r % 256 != 0) return false;
    if (r == d) return d <= 2048;                  // full keys: d = 256 * (1..8)
    const int kcpl = r / 256;                      // sliced keys: r = 256 * {1,2,4,8}
    return d <= 4096 && (kcpl == 1 || kcpl == 2 || kcpl == 4 || kcpl == 8);
}

}  // namespace ar

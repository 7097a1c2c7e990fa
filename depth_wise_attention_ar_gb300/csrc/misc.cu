// Bank append (+ inverse RMS), the fixed-order dq/dg reduction, the device
// error word, and the dtype dispatch of the routing launches.
#include "common.cuh"
#include "launch_util.cuh"

namespace ar {

template <typename T> cudaError_t dispatch_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps);
template <typename T> cudaError_t dispatch_lr_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_lr_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps);
template <typename T> cudaError_t dispatch_coop_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_coop_bwd(const RouteArgs *a, cudaStream_t s, int *grid_rows);

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
                                                     int norm_full, float eps, int src_tok_stride)
{
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nch = d / 8;
    const int c0 = norm_full ? 0 : (d - r) / 8;
    const float inv_w = 1.0f / (float)(norm_full ? d : r);
    const bool write = (src != dst) || prev != nullptr || src_tok_stride != d;
    for (int64_t t = w0; t < TT; t += nw) {
        const T *s = src + t * src_tok_stride;
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
                          cudaStream_t s, bool broadcast)
{
    const int stride = broadcast ? 0 : d;
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
            static_cast<__nv_bfloat16 *>(dst), inv_col, T, d, r, inv_ld, norm_full, eps, stride);
    else
        append_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(src),
                                                  static_cast<const float *>(prev),
                                                  static_cast<float *>(dst), inv_col, T, d, r,
                                                  inv_ld, norm_full, eps, stride);
    return cudaGetLastError();
}

// ---- gradient fold (block-sum fan-out) -----------------------------------------
// dst += src over one [T, d] pair of fp32 gradient rows (dst = src when dst
// has not been written since zero_grad; dst = 0 when neither has). A block
// partial-sum version t+1 = version t + o_{t+1} passes its whole adjoint on to
// version t ("Low-Rank Attention Residuals", Appendix B.4: every write of a
// block receives the block sum's adjoint).
__global__ void __launch_bounds__(256) grad_fold_kernel(float *dst, const float *src, int64_t n4,
                                                        int mode)
{
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mode & 1) v = s4[i];                  // src has content
        if (mode & 2) {                           // dst has content
            const float4 o = d4[i];
            v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
        }
        d4[i] = v;
    }
}

cudaError_t launch_grad_fold(float *dst, const float *src, int64_t n, bool src_valid,
                             bool dst_valid, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    int grid = 0;
    cudaError_t e = persistent_grid(reinterpret_cast<const void *>(&grad_fold_kernel), 256, 0, &grid);
    if (e != cudaSuccess) return e;
    const int64_t n4 = n / 4;
    const int64_t need = (n4 + 255) / 256;
    if (need < grid) grid = (int)need;
    grad_fold_kernel<<<grid, 256, 0, s>>>(dst, src, n4, (src_valid ? 1 : 0) | (dst_valid ? 2 : 0));
    return cudaGetLastError();
}

// ---- gradient of a broadcast row ----------------------------------------------
// out[c] = sum_t grad[t, c] over one [T, d] fp32 gradient row: the gradient of
// a source that is the same vector for every token (the learnable null source
// of the delta form, "Multi-Head Attention Residuals", Sec. 3.3). One block per
// 32 columns; warp w sums tokens w, w + 8, ..., then the 8 warps in order.
__global__ void __launch_bounds__(256) token_sum_kernel(const float *grad, int64_t TT, int d,
                                                        float *out)
{
    __shared__ float part[8][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (c < d)
        for (int64_t t = w; t < TT; t += 8) s += grad[t * d + c];
    part[w][lane] = s;
    __syncthreads();
    if (w == 0 && c < d) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) t += part[k][lane];
        out[c] = t;
    }
}

cudaError_t launch_token_sum(const float *grad, int64_t T, int d, float *out, cudaStream_t s)
{
    token_sum_kernel<<<(d + 31) / 32, 256, 0, s>>>(grad, T, d, out);
    return cudaGetLastError();
}

// ---- merge of two partial reads (two-phase block inference) --------------------
// For two disjoint source sets A and B of one site, with per-head results
// (out_A, lse_A) and (out_B, lse_B), the read over A u B is
//   lse = m + log(e^(lse_A - m) + e^(lse_B - m)),  m = max(lse_A, lse_B)
//   out = (e^(lse_A - lse) out_A + e^(lse_B - lse) out_B)   on each head's slice
// ("Low-Rank Attention Residuals", Sec. 3.4: inter-block and intra-block
// results merge with an online-softmax update). One warp per token.
template <typename T>
__global__ void __launch_bounds__(256) merge_kernel(const T *oa, const float *la, const T *ob,
                                                    const float *lb, T *out, float *lse,
                                                    int64_t TT, int d, int H)
{
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int K = d / H, nch = d / 8;
    for (int64_t t = w0; t < TT; t += nw) {
        for (int c = lane; c < nch; c += 32) {
            const int h = (c * 8) / K;
            const float a = la[t * H + h], b = lb[t * H + h];
            const float m = fmaxf(a, b);
            const float ea = exp2f((a - m) * kLog2e), eb = exp2f((b - m) * kLog2e);
            const float inv = 1.f / (ea + eb);
            float x[8], y[8], z[8];
            ld_chunk_g(oa + t * d + c * 8, x);
            ld_chunk_g(ob + t * d + c * 8, y);
#pragma unroll
            for (int e = 0; e < 8; ++e) z[e] = fmaf(ea * inv, x[e], eb * inv * y[e]);
            st_chunk_g(out + t * d + c * 8, z);
        }
        for (int h = lane; h < H; h += 32) {
            const float a = la[t * H + h], b = lb[t * H + h];
            const float m = fmaxf(a, b);
            lse[t * H + h] = m + log2f(exp2f((a - m) * kLog2e) + exp2f((b - m) * kLog2e)) * kLn2;
        }
    }
}

cudaError_t launch_merge(const void *oa, const float *la, const void *ob, const float *lb,
                         void *out, float *lse, int64_t T, int d, int H, ar_dtype dt, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const void *k = dt == AR_BF16 ? reinterpret_cast<const void *>(&merge_kernel<__nv_bfloat16>)
                                  : reinterpret_cast<const void *>(&merge_kernel<float>);
    int grid = 0;
    cudaError_t e = persistent_grid(k, 256, 0, &grid);
    if (e != cudaSuccess) return e;
    const int64_t need = (T + 7) / 8;
    if (need < grid) grid = (int)need;
    if (dt == AR_BF16)
        merge_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(oa), la, static_cast<const __nv_bfloat16 *>(ob), lb,
            static_cast<__nv_bfloat16 *>(out), lse, T, d, H);
    else
        merge_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(oa), la,
                                                 static_cast<const float *>(ob), lb,
                                                 static_cast<float *>(out), lse, T, d, H);
    return cudaGetLastError();
}

// ---- dq / dg -----------------------------------------------------------------
// dq_c = g_c * sum_w ws[w, c], dg_c = q_c * sum_w ws[w, c]; the sum over the
// backward's warps runs in a fixed order (8 strided groups, then the groups
// in order), so repeated runs give identical bits.
__global__ void __launch_bounds__(256) dqdg_reduce_kernel(const float *ws, int rows, int r,
                                                          const float *q, const float *g,
                                                          float *dq, float *dg, float *dalpha)
{
    __shared__ float part[8][33];
    if (dalpha && blockIdx.x == 0) {
        // dL/dalpha of the delta form: the rows * 4 tail partials, fixed order
        __shared__ float red[256];
        const float *tail = ws + (int64_t)rows * r;
        float s = 0.f;
        for (int k = threadIdx.x; k < rows * 4; k += 256) s += tail[k];
        red[threadIdx.x] = s;
        __syncthreads();
        for (int o = 128; o > 0; o >>= 1) {
            if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
            __syncthreads();
        }
        if (threadIdx.x == 0) *dalpha = red[0];
        __syncthreads();
    }
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
                               float *dq, float *dg, float *dalpha, cudaStream_t s)
{
    dqdg_reduce_kernel<<<(r + 31) / 32, 256, 0, s>>>(ws, rows, r, q, g, dq, dg, dalpha);
    return cudaGetLastError();
}

// ---- dtype / shape dispatch ----------------------------------------------------
// r = d, d <= 2048: one warp per token (online softmax, register-resident).
// d > 2048, or r < d with d a multiple of 1024: four warps share each row.
// Other sliced-key shapes (d <= 4096): one warp per token, two-sweep forward.
enum class Family { kFull, kCoop, kSliced, kNone };

static Family family_of(int d, int r, int H)
{
    if (H < 1 || d <= 0 || r <= 0 || r > d || d % 256 != 0 || r % 8 != 0) return Family::kNone;
    const bool pow2_h = H <= 32 && (32 % H) == 0;
    if (r == d && d <= 2048 && pow2_h) return Family::kFull;
    if (r % 256 == 0 && coop_supported(d, r, H)) return Family::kCoop;
    // one warp per token, two sweeps: any key width with whole 8-column chunks
    // per head (r = d included, for widths the other families leave out)
    if (d <= 4096 && pow2_h && (r / H) % 8 == 0 && (r + 255) / 256 <= 16) return Family::kSliced;
    return Family::kNone;
}

cudaError_t launch_route_fwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s)
{
    const bool bf = dt == AR_BF16;
    switch (family_of(a.d, a.r, a.H)) {
    case Family::kFull: return bf ? dispatch_fwd<__nv_bfloat16>(a, s) : dispatch_fwd<float>(a, s);
    case Family::kCoop:
        return bf ? dispatch_coop_fwd<__nv_bfloat16>(a, s) : dispatch_coop_fwd<float>(a, s);
    case Family::kSliced:
        return bf ? dispatch_lr_fwd<__nv_bfloat16>(a, s) : dispatch_lr_fwd<float>(a, s);
    default: return cudaErrorNotSupported;
    }
}

static cudaError_t bwd_any(const RouteArgs &a, ar_dtype dt, cudaStream_t s, int *rows)
{
    const bool bf = dt == AR_BF16;
    switch (family_of(a.d, a.r, a.H)) {
    case Family::kFull:
        return bf ? dispatch_bwd<__nv_bfloat16>(&a, s, rows) : dispatch_bwd<float>(&a, s, rows);
    case Family::kCoop:
        return bf ? dispatch_coop_bwd<__nv_bfloat16>(&a, s, rows)
                  : dispatch_coop_bwd<float>(&a, s, rows);
    case Family::kSliced:
        return bf ? dispatch_lr_bwd<__nv_bfloat16>(&a, s, rows) : dispatch_lr_bwd<float>(&a, s, rows);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_route_bwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s)
{
    return bwd_any(a, dt, s, nullptr);
}

cudaError_t route_bwd_grid(const RouteArgs &a, ar_dtype dt, int *grid_rows)
{
    return bwd_any(a, dt, nullptr, grid_rows);
}

bool fused_shape_supported(int d, int r, int H) { return family_of(d, r, H) != Family::kNone; }

bool delta_supported(int d, int r, int H)
{
    const Family f = family_of(d, r, H);
    return f == Family::kFull || f == Family::kCoop;
}

}  // namespace ar

// Bank append (+ inverse RMS), the fixed-order dq/dg reduction, the device
// error word, and the dtype dispatch of the routing launches.
#include "common.cuh"
#include "launch_util.cuh"
#include "shapes.h"

#include <cooperative_groups.h>

#include <mutex>

namespace ar {

namespace cg = cooperative_groups;

template <typename T> cudaError_t dispatch_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps);
template <typename T> cudaError_t dispatch_lr_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_fwd_sk(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_fwd_multi(const MultiArgs &m, cudaStream_t s);
template <typename T> cudaError_t dispatch_lr_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps);
template <typename T> cudaError_t dispatch_coop_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_coop_bwd(const RouteArgs *a, cudaStream_t s, int *grid_rows);
template <typename T> cudaError_t dispatch_generic_fwd(const RouteArgs &a, cudaStream_t s);
template <typename T> cudaError_t dispatch_generic_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps);
template <typename T> cudaError_t dispatch_coupling(const RouteArgs &a, float *S, cudaStream_t s);

// Device error word; kernels get its address as an argument.
__device__ unsigned int g_device_error = 0;

unsigned int *device_error_word()
{
    // cached per device (devices 0..63): the symbol lookup is done once,
    // outside any capture; the lock keeps first calls from several host
    // threads off each other's entries
    static std::mutex mu;
    static unsigned int *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int *>(p);
    }
    return cache[dev];
}

#ifdef AR_CHECKED
// The checked build's record of its first refused access: [taken, address,
// kind << 32 | bytes].
__device__ unsigned long long g_check_fault[3] = {0ull, 0ull, 0ull};

unsigned long long *device_check_fault()
{
    static std::mutex mu;
    static unsigned long long *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_check_fault) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned long long *>(p);
    }
    return cache[dev];
}
#endif

// ---- append ----------------------------------------------------------------
// One warp per token. new = src (copied only when src is not the slot
// itself), or prev + src in fp32 rounded once to the storage dtype (block
// partial sums, "Low-Rank Attention Residuals" Sec. 3.3 / Figure 11). The
// inverse RMS is taken over the stored (rounded) values of the RMS
// coordinates: the last r ("Low-Rank Attention Residuals" Eq. 11/13), or all
// d for the full-width norm ("Multi-Head Attention Residuals" Appendix E).
// The source is a strided [T, d] view: element (t, c) at src[t * ld + c * es]
// (ld = 0 broadcasts one vector to every token).
//   kInPlace: the row already sits in its slot; 16-byte reads of its RMS
//             chunks only.
//   kCopy   : 16-byte reads of src (and prev), 16-byte stores (d and the
//             first RMS column multiples of 8, es = 1, aligned rows).
//   kScalar : anything else, one element at a time.
// kScalar walks the row in the same 8-column chunks and lane order as the
// 16-byte mode it stands in for, so a strided source gives the same bits as
// a contiguous one.
enum AppendMode { kInPlace = 0, kCopy = 1, kScalar = 2 };

__device__ __forceinline__ float round_bf16(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

template <typename T, int MODE>
__global__ void __launch_bounds__(256) append_kernel(const T *src, const T *prev, T *dst, float *inv,
                                                     int64_t TT, int d, int r, int inv_ld,
                                                     int norm_full, float eps, int64_t ld,
                                                     int64_t es, bool in_place AR_CHK_PARAM)
{
    AR_CHK_ENTER_PARAM();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nch = (d + 7) / 8;
    const int col0 = norm_full ? 0 : d - r;  // first RMS coordinate
    const float inv_w = 1.0f / (float)(norm_full ? d : r);
    for (int64_t t = w0; t < TT; t += nw) {
        const T *s = src + t * ld;
        T *o = dst + t * d;
        float ss = 0.f;
        if constexpr (MODE == kInPlace) {
            for (int c = col0 / 8 + lane; c < nch; c += 32) {
                float x[8];
                ld_chunk_g(o + c * 8, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
            }
        } else if constexpr (MODE == kCopy) {
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
                if (c * 8 >= col0) {
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
            for (int c = (in_place ? col0 / 8 : 0) + lane; c < nch; c += 32) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int col = c * 8 + e;
                    if (col < d) {
                        float v = to_f32(in_place ? ld_chk_t(o + col) : ld_chk_t(s + col * es));
                        if (prev) v += to_f32(ld_chk_t(prev + (t * d + col)));
                        if (!in_place) st_elem(o + col, v);
                        // square the stored (rounded) value
                        const float vr = sizeof(T) == 2 ? round_bf16(v) : v;
                        if (col >= col0) ss = fmaf(vr, vr, ss);
                    }
                }
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) st_chk_t(inv + t * inv_ld, rsqrtf(fmaf(ss, inv_w, eps)));
    }
}

#ifdef AR_CHECKED
// The table a launch passes when its caller gave none: not checked.
static const RouteArgs &chk_or_off(const RouteArgs *chk)
{
    static RouteArgs off = [] {
        RouteArgs a{};
        a.chk.off = 1;
        return a;
    }();
    return chk ? *chk : off;
}
#endif

template <typename E>
static cudaError_t append_t(const void *src, const void *prev, void *dst, float *inv_col, int64_t T,
                            int d, int r, int inv_ld, int norm_full, float eps, int64_t ld,
                            int64_t es, cudaStream_t s, const RouteArgs *chk)
{
    (void)chk;
    const bool in_place = src == dst && prev == nullptr && ld == d && es == 1;
    const uintptr_t al = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                         reinterpret_cast<uintptr_t>(prev);
    const int col0 = norm_full ? 0 : d - r;
    const bool vec = d % 8 == 0 && col0 % 8 == 0 && es == 1 &&
                     (ld * (int64_t)sizeof(E)) % 16 == 0 && (al & 15) == 0;
    const int mode = !vec ? kScalar : in_place ? kInPlace : kCopy;
    const void *k = mode == kInPlace ? reinterpret_cast<const void *>(&append_kernel<E, kInPlace>)
                    : mode == kCopy  ? reinterpret_cast<const void *>(&append_kernel<E, kCopy>)
                                     : reinterpret_cast<const void *>(&append_kernel<E, kScalar>);
    int grid = 0;
    cudaError_t e = persistent_grid(k, 256, 0, &grid);
    if (e != cudaSuccess) return e;
    const int64_t need = (T + 7) / 8;
    if (need < grid) grid = (int)need;
    const E *sp = static_cast<const E *>(src), *pp = static_cast<const E *>(prev);
    E *dp = static_cast<E *>(dst);
    if (mode == kInPlace)
        append_kernel<E, kInPlace><<<grid, 256, 0, s>>>(sp, pp, dp, inv_col, T, d, r, inv_ld,
                                                        norm_full, eps, ld, es,
                                                        in_place AR_CHK_PASS(chk_or_off(chk)));
    else if (mode == kCopy)
        append_kernel<E, kCopy><<<grid, 256, 0, s>>>(sp, pp, dp, inv_col, T, d, r, inv_ld,
                                                     norm_full, eps, ld, es,
                                                     in_place AR_CHK_PASS(chk_or_off(chk)));
    else
        append_kernel<E, kScalar><<<grid, 256, 0, s>>>(sp, pp, dp, inv_col, T, d, r, inv_ld,
                                                       norm_full, eps, ld, es,
                                                       in_place AR_CHK_PASS(chk_or_off(chk)));
    return cudaGetLastError();
}

cudaError_t launch_append(const void *src, const void *prev, void *dst, float *inv_col, int64_t T,
                          int d, int r, int inv_ld, int norm_full, float eps, ar_dtype dt,
                          cudaStream_t s, int64_t ld, int64_t es, const RouteArgs *chk)
{
    if (T == 0) return cudaSuccess;
    return dt == AR_BF16 ? append_t<__nv_bfloat16>(src, prev, dst, inv_col, T, d, r, inv_ld,
                                                   norm_full, eps, ld, es, s, chk)
                         : append_t<float>(src, prev, dst, inv_col, T, d, r, inv_ld, norm_full,
                                           eps, ld, es, s, chk);
}

// ---- gradient fold (block-sum fan-out) -----------------------------------------
// dst += src over one [T, d] pair of fp32 gradient rows (dst = src when dst
// has not been written since zero_grad; dst = 0 when neither has). A block
// partial-sum version t+1 = version t + o_{t+1} passes its whole adjoint on to
// version t ("Low-Rank Attention Residuals", Appendix B.4: every write of a
// block receives the block sum's adjoint).
__global__ void __launch_bounds__(256) grad_fold_scalar_kernel(float *dst, const float *src,
                                                               int64_t n, int mode AR_CHK_PARAM)
{
    AR_CHK_ENTER_PARAM();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        st_chk_t(dst + i, ((mode & 1) ? ld_chk_t(src + i) : 0.f) + ((mode & 2) ? ld_chk_t(dst + i) : 0.f));
}

__global__ void __launch_bounds__(256) grad_fold_kernel(float *dst, const float *src, int64_t n4,
                                                        int mode AR_CHK_PARAM)
{
    AR_CHK_ENTER_PARAM();
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mode & 1) v = ld_chk_t(s4 + i);       // src has content
        if (mode & 2) {                           // dst has content
            const float4 o = ld_chk_t(d4 + i);
            v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
        }
        st_chk_t(d4 + i, v);
    }
}

cudaError_t launch_grad_fold(float *dst, const float *src, int64_t n, bool src_valid,
                             bool dst_valid, cudaStream_t s, const RouteArgs *chk)
{
    (void)chk;
    if (n == 0) return cudaSuccess;
    const int mode = (src_valid ? 1 : 0) | (dst_valid ? 2 : 0);
    int grid = 0;
    const uintptr_t al = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src);
    if (n % 4 != 0 || (al & 15) != 0) {  // rows of an unaligned width
        cudaError_t e = persistent_grid(reinterpret_cast<const void *>(&grad_fold_scalar_kernel),
                                        256, 0, &grid);
        if (e != cudaSuccess) return e;
        const int64_t need = (n + 255) / 256;
        if (need < grid) grid = (int)need;
        grad_fold_scalar_kernel<<<grid, 256, 0, s>>>(dst, src, n, mode AR_CHK_PASS(chk_or_off(chk)));
        return cudaGetLastError();
    }
    cudaError_t e = persistent_grid(reinterpret_cast<const void *>(&grad_fold_kernel), 256, 0, &grid);
    if (e != cudaSuccess) return e;
    const int64_t n4 = n / 4;
    const int64_t need = (n4 + 255) / 256;
    if (need < grid) grid = (int)need;
    grad_fold_kernel<<<grid, 256, 0, s>>>(dst, src, n4, mode AR_CHK_PASS(chk_or_off(chk)));
    return cudaGetLastError();
}

// ---- gradient of a broadcast row ----------------------------------------------
// out[c] = sum_t grad[t, c] over one [T, d] fp32 gradient row: the gradient of
// a source that is the same vector for every token (the learnable null source
// of the delta form, "Multi-Head Attention Residuals", Sec. 3.3). One block per
// 32 columns; warp w sums tokens w, w + 8, ..., then the 8 warps in order.
__global__ void __launch_bounds__(256) token_sum_kernel(const float *grad, int64_t TT, int d,
                                                        float *out AR_CHK_PARAM)
{
    AR_CHK_ENTER_PARAM();
    __shared__ float part[8][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (c < d)
        for (int64_t t = w; t < TT; t += 8) s += ld_chk_t(grad + (t * d + c));
    part[w][lane] = s;
    __syncthreads();
    if (w == 0 && c < d) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) t += part[k][lane];
        st_chk_t(out + c, t);
    }
}

cudaError_t launch_token_sum(const float *grad, int64_t T, int d, float *out, cudaStream_t s,
                             const RouteArgs *chk)
{
    (void)chk;
    token_sum_kernel<<<(d + 31) / 32, 256, 0, s>>>(grad, T, d, out AR_CHK_PASS(chk_or_off(chk)));
    return cudaGetLastError();
}

// ---- merge of two partial reads (two-phase block inference) --------------------
// For two disjoint source sets A and B of one site, with per-head results
// (out_A, lse_A) and (out_B, lse_B), the read over A u B is
//   lse = m + log(e^(lse_A - m) + e^(lse_B - m)),  m = max(lse_A, lse_B)
//   out = (e^(lse_A - lse) out_A + e^(lse_B - lse) out_B)   on each head's slice
// ("Low-Rank Attention Residuals", Sec. 3.4: two-phase block inference
// combines the read over the finished blocks with the read over the partial
// sum by their log-sum-exp, as one step of an online softmax). One warp per
// token.
// VEC: 8-column chunks (d and d/H multiples of 8, aligned rows); otherwise
// one column at a time, with the same arithmetic per element.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) merge_kernel(const T *oa, const float *la, const T *ob,
                                                    const float *lb, T *out, float *lse,
                                                    int64_t TT, int d, int H AR_CHK_PARAM)
{
    AR_CHK_ENTER_PARAM();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int K = d / H, nch = VEC ? d / 8 : d;
    for (int64_t t = w0; t < TT; t += nw) {
        for (int c = lane; c < nch; c += 32) {
            const int h = (VEC ? c * 8 : c) / K;
            const float a = ld_chk_t(la + (t * H + h)), b = ld_chk_t(lb + (t * H + h));
            const float m = fmaxf(a, b);
            const float ea = exp2f((a - m) * kLog2e), eb = exp2f((b - m) * kLog2e);
            const float inv = 1.f / (ea + eb);
            if constexpr (VEC) {
                float x[8], y[8], z[8];
                ld_chunk_g(oa + t * d + c * 8, x);
                ld_chunk_g(ob + t * d + c * 8, y);
#pragma unroll
                for (int e = 0; e < 8; ++e) z[e] = fmaf(ea * inv, x[e], eb * inv * y[e]);
                st_chunk_g(out + t * d + c * 8, z);
            } else {
                const float x = to_f32(ld_chk_t(oa + (t * d + c))), y = to_f32(ld_chk_t(ob + (t * d + c)));
                st_elem(out + t * d + c, fmaf(ea * inv, x, eb * inv * y));
            }
        }
        for (int h = lane; h < H; h += 32) {
            const float a = ld_chk_t(la + (t * H + h)), b = ld_chk_t(lb + (t * H + h));
            const float m = fmaxf(a, b);
            st_chk_t(lse + (t * H + h), m + log2f(exp2f((a - m) * kLog2e) + exp2f((b - m) * kLog2e)) * kLn2);
        }
    }
}

template <typename E>
static cudaError_t merge_t(const void *oa, const float *la, const void *ob, const float *lb,
                           void *out, float *lse, int64_t T, int d, int H, cudaStream_t s,
                           const RouteArgs *chk)
{
    (void)chk;
    const uintptr_t al = reinterpret_cast<uintptr_t>(oa) | reinterpret_cast<uintptr_t>(ob) |
                         reinterpret_cast<uintptr_t>(out);
    const bool vec = d % 8 == 0 && (d / H) % 8 == 0 && (al & 15) == 0;
    const void *k = vec ? reinterpret_cast<const void *>(&merge_kernel<E, true>)
                        : reinterpret_cast<const void *>(&merge_kernel<E, false>);
    int grid = 0;
    cudaError_t e = persistent_grid(k, 256, 0, &grid);
    if (e != cudaSuccess) return e;
    const int64_t need = (T + 7) / 8;
    if (need < grid) grid = (int)need;
    const E *a = static_cast<const E *>(oa), *b = static_cast<const E *>(ob);
    E *o = static_cast<E *>(out);
    if (vec)
        merge_kernel<E, true><<<grid, 256, 0, s>>>(a, la, b, lb, o, lse, T, d,
                                                   H AR_CHK_PASS(chk_or_off(chk)));
    else
        merge_kernel<E, false><<<grid, 256, 0, s>>>(a, la, b, lb, o, lse, T, d,
                                                    H AR_CHK_PASS(chk_or_off(chk)));
    return cudaGetLastError();
}

cudaError_t launch_merge(const void *oa, const float *la, const void *ob, const float *lb,
                         void *out, float *lse, int64_t T, int d, int H, ar_dtype dt, cudaStream_t s,
                         const RouteArgs *chk)
{
    if (T == 0) return cudaSuccess;
    return dt == AR_BF16 ? merge_t<__nv_bfloat16>(oa, la, ob, lb, out, lse, T, d, H, s, chk)
                         : merge_t<float>(oa, la, ob, lb, out, lse, T, d, H, s, chk);
}

// ---- dq / dg -----------------------------------------------------------------
// dq_c = g_c * sum_w ws[w, c], dg_c = q_c * sum_w ws[w, c] over the
// backward's partial rows w (one per block of the backward grid).
//
// One cluster of kRedCtas CTAs per tile of 32 * V columns (V = 4: float4
// columns when r is a multiple of 4). The cluster's 8 x 16 warps take the
// rows round-robin, each with eight running sums: a warp's rows (about ten
// for a persistent backward grid) arrive in two rounds of eight loads in
// flight. A CTA adds its warps' sums in warp order in shared
// memory, and CTA 0 adds the CTAs' sums in rank order through distributed
// shared memory. Every sum has a fixed order, so repeated runs give identical
// bits.
constexpr int kRedCtas = 8;
constexpr int kRedWarps = 16;

constexpr int kRedSums = 8;   // running sums (and loads in flight) per lane
static_assert(kRedSums == 8, "the sums are combined as a fixed tree of eight");

template <int V>
__device__ __forceinline__ void red_load(const float *p, float (&x)[V])
{
    if constexpr (V == 4) {
        AR_GUARD_G(p, 16, false, 16, x[0] = x[1] = x[2] = x[3] = 0.f; return)
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(p));
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    } else {
        AR_GUARD_G(p, 4, false, 4, x[0] = 0.f; return)
        x[0] = __ldcg(p);
    }
}

template <int V>
__global__ void __cluster_dims__(kRedCtas, 1, 1) __launch_bounds__(kRedWarps * 32)
    dqdg_reduce_kernel(const float *__restrict__ ws, int rows, int r, const float *q, int64_t qs,
                       const float *g, int64_t gs, float *dq, float *dg,
                       float *dalpha AR_CHK_PARAM)
{
    AR_CHK_ENTER_PARAM();
    __shared__ float part[kRedWarps][32 * V];
    __shared__ float cta_sum[32 * V];
    __shared__ float red[kRedWarps * 32];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c0 = (blockIdx.y * 32 + lane) * V;   // this lane's first column
    const bool valid = c0 < r;
    constexpr int stride = kRedCtas * kRedWarps;

    float s[kRedSums][V];
#pragma unroll
    for (int u = 0; u < kRedSums; ++u)
#pragma unroll
        for (int e = 0; e < V; ++e) s[u][e] = 0.f;
    if (valid) {
        // rounds of kRedSums rows (w + u * stride, u = 0 .. kRedSums - 1), all
        // loads of a round issued before the first add; rows past the end
        // add zero
        for (int w = rank * kRedWarps + warp; w < rows; w += kRedSums * stride) {
            float x[kRedSums][V];
#pragma unroll
            for (int u = 0; u < kRedSums; ++u) {
#pragma unroll
                for (int e = 0; e < V; ++e) x[u][e] = 0.f;
                if (w + u * stride < rows) red_load<V>(ws + (int64_t)(w + u * stride) * r + c0, x[u]);
            }
#pragma unroll
            for (int u = 0; u < kRedSums; ++u)
#pragma unroll
                for (int e = 0; e < V; ++e) s[u][e] += x[u][e];
        }
    }
#pragma unroll
    for (int e = 0; e < V; ++e)
        part[warp][lane * V + e] = ((s[0][e] + s[1][e]) + (s[2][e] + s[3][e])) +
                                   ((s[4][e] + s[5][e]) + (s[6][e] + s[7][e]));
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int e = 0; e < V; ++e) {
            float t = 0.f;
#pragma unroll
            for (int k = 0; k < kRedWarps; ++k) t += part[k][lane * V + e];
            cta_sum[lane * V + e] = t;
        }
    }
    cl.sync();
    if (rank == 0 && warp == 0 && valid) {
        float t[V];
#pragma unroll
        for (int e = 0; e < V; ++e) t[e] = 0.f;
#pragma unroll
        for (int k = 0; k < kRedCtas; ++k) {
            const float *rem = cl.map_shared_rank(cta_sum, k);
#pragma unroll
            for (int e = 0; e < V; ++e) t[e] += rem[lane * V + e];
        }
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const int c = c0 + e;
            st_chk_t(dq + c * qs, (g ? ld_chk_t(g + c * gs) : 1.0f) * t[e]);
            if (dg) st_chk_t(dg + c * gs, ld_chk_t(q + c * qs) * t[e]);
        }
    }
    if (dalpha && blockIdx.y == 0 && rank == 1) {
        // dL/dalpha of the delta form: the rows * 4 tail partials, fixed order
        const float *tail = ws + (int64_t)rows * r;
        float a = 0.f;
        for (int k = threadIdx.x; k < rows * 4; k += kRedWarps * 32) a += ld_chk_t(tail + k);
        red[threadIdx.x] = a;
        __syncthreads();
        for (int o = kRedWarps * 16; o > 0; o >>= 1) {
            if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
            __syncthreads();
        }
        if (threadIdx.x == 0) st_chk_t(dalpha, red[0]);
    }
    // no CTA leaves while CTA 0 may still read its shared memory
    cl.sync();
}

cudaError_t launch_dqdg_reduce(const float *ws, int rows, int r, const float *q, int64_t q_stride,
                               const float *g, int64_t g_stride, float *dq, float *dg,
                               float *dalpha, cudaStream_t s, const RouteArgs *chk)
{
    (void)chk;
    if (r % 4 == 0) {
        const dim3 grid(kRedCtas, (r / 4 + 31) / 32);
        dqdg_reduce_kernel<4><<<grid, kRedWarps * 32, 0, s>>>(ws, rows, r, q, q_stride, g,
                                                             g_stride, dq, dg,
                                                             dalpha AR_CHK_PASS(chk_or_off(chk)));
    } else {
        const dim3 grid(kRedCtas, (r + 31) / 32);
        dqdg_reduce_kernel<1><<<grid, kRedWarps * 32, 0, s>>>(ws, rows, r, q, q_stride, g,
                                                             g_stride, dq, dg,
                                                             dalpha AR_CHK_PASS(chk_or_off(chk)));
    }
    return cudaGetLastError();
}

// ---- dtype / shape dispatch (family rules in shapes.h) ---------------------------
cudaError_t launch_route_fwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s)
{
    const bool bf = dt == AR_BF16;
    switch (family_of(a.d, a.r, a.H, a.n_src, bf ? 2 : 4, a.has_bias != 0)) {
    case Family::kFull: return bf ? dispatch_fwd<__nv_bfloat16>(a, s) : dispatch_fwd<float>(a, s);
    case Family::kCoop:
        return bf ? dispatch_coop_fwd<__nv_bfloat16>(a, s) : dispatch_coop_fwd<float>(a, s);
    case Family::kSliced:
        // rows up to 2560 wide: one pass with the accumulator in registers;
        // wider rows: two sweeps with the key tails cached in shared memory
        if (a.d / 256 <= 10)
            return bf ? dispatch_fwd_sk<__nv_bfloat16>(a, s) : dispatch_fwd_sk<float>(a, s);
        return bf ? dispatch_lr_fwd<__nv_bfloat16>(a, s) : dispatch_lr_fwd<float>(a, s);
    case Family::kGeneric:
        return bf ? dispatch_generic_fwd<__nv_bfloat16>(a, s) : dispatch_generic_fwd<float>(a, s);
    default: return cudaErrorNotSupported;
    }
}

static cudaError_t bwd_any(const RouteArgs &a, ar_dtype dt, cudaStream_t s, int *rows)
{
    const bool bf = dt == AR_BF16;
    switch (family_of(a.d, a.r, a.H, a.n_src, bf ? 2 : 4, a.has_bias != 0)) {
    case Family::kFull:
        return bf ? dispatch_bwd<__nv_bfloat16>(&a, s, rows) : dispatch_bwd<float>(&a, s, rows);
    case Family::kCoop:
        return bf ? dispatch_coop_bwd<__nv_bfloat16>(&a, s, rows)
                  : dispatch_coop_bwd<float>(&a, s, rows);
    case Family::kSliced:
        return bf ? dispatch_lr_bwd<__nv_bfloat16>(&a, s, rows) : dispatch_lr_bwd<float>(&a, s, rows);
    case Family::kGeneric:
        return bf ? dispatch_generic_bwd<__nv_bfloat16>(&a, s, rows)
                  : dispatch_generic_bwd<float>(&a, s, rows);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_route_coupling(const RouteArgs &a, float *S, ar_dtype dt, cudaStream_t s)
{
    return dt == AR_BF16 ? dispatch_coupling<__nv_bfloat16>(a, S, s) : dispatch_coupling<float>(a, S, s);
}

cudaError_t launch_route_bwd(const RouteArgs &a, ar_dtype dt, cudaStream_t s)
{
    return bwd_any(a, dt, s, nullptr);
}

cudaError_t route_bwd_grid(const RouteArgs &a, ar_dtype dt, int *grid_rows)
{
    return bwd_any(a, dt, nullptr, grid_rows);
}

bool fwd_fuses_append(const RouteArgs &a, ar_dtype dt, bool in_place)
{
    if (a.has_bias || a.partial) return false;
    const Family f = family_of(a.d, a.r, a.H, a.n_src, dt == AR_BF16 ? 2 : 4, false);
    if (f == Family::kCoop) return true;
    // one-warp kernels, rows up to 1024 wide: at 1280 the fused forward measured
    // slower than the separate append (1B forward phase 18.02 -> 18.46 ms)
    return in_place && f == Family::kFull && a.r == a.d && a.d <= 1024;
}

// One block per token with one lane per 8-column chunk: d a multiple of 256
// up to 4096, whole chunks per value and key head.
cudaError_t launch_route_fwd_multi(const MultiArgs &m, ar_dtype dt, cudaStream_t s)
{
    const RouteArgs &a = m.base;
    if (a.d % 256 != 0 || a.d > 4096 || (a.d / a.H) % 8 != 0 || (a.r / a.H) % 8 != 0)
        return cudaErrorNotSupported;
    if (dt == AR_BF16) {
        // tensor cores where the shape fits them, else the CUDA-core kernel
        const cudaError_t e = dispatch_fwd_multi_mma(m, s);
        if (e != cudaErrorNotSupported) return e;
        return dispatch_fwd_multi<__nv_bfloat16>(m, s);
    }
    return dispatch_fwd_multi<float>(m, s);
}

bool route_supported(int d, int r, int H, int n_src, ar_dtype dt, bool repeats)
{
    return family_of(d, r, H, n_src, dt == AR_BF16 ? 2 : 4, repeats) != Family::kNone;
}

cudaError_t generic_bwd_rows(int *rows)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    *rows = sms * kGenBlocksPerSm;
    return cudaSuccess;
}

}  // namespace ar

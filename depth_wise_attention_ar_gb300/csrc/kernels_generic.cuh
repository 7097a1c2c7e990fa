// Routing kernels for every shape the tiled families leave out: any width d,
// any key width r <= d, any head count H dividing both ("Low-Rank Attention
// Residuals", Appendix I: the operator tiles unaligned widths and ranks, and
// is checked at d = 513). Same arithmetic as the tiled kernels (scores
// z = inv * <q g, key slice>, softmax over the listed rows per head, mix of
// the value slices; the single-pass backward with the coupling term read from
// the forward output), with scalar element accesses: a token's row starts at
// (row * T + t) * d elements, which for such widths carries no 16-byte
// alignment, so neither bulk copies nor vector loads apply.
//
// One warp per token, tokens strided over a fixed grid. Lanes stride over
// the coordinates of a head slice for the dot products (one warp reduction
// per head), then over the row for the mix / gradient pass, with the rows
// inner, so that every load instruction reads 32 consecutive elements of one
// row. Per-warp shared memory holds the site's scores or weights [N, H]; the
// block shares q*g over the key coordinates. The backward also keeps its
// warp's dq/dg partial sums (one per key coordinate) in shared memory; at the
// end each block adds its warps' sums, in order, into one workspace row.
// Sites that list a row k > 1 times also run here: the row enters once with
// log k added to its score (the softmax over the list), a term the tiled
// kernels leave out of their inner loops.
#pragma once

#include "common.cuh"
#include "launch_util.cuh"
#include "shapes.h"

namespace ar {

template <typename T> __device__ __forceinline__ float gen_ld(const T *p);
template <> __device__ __forceinline__ float gen_ld<float>(const float *p) { return ldg_chk(p); }
template <> __device__ __forceinline__ float gen_ld<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    AR_GUARD_G(p, 2, false, 2, return 0.f)
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __uint_as_float((uint32_t)u << 16);
}

__device__ __forceinline__ float gen_qg(const RouteArgs &a, int c)
{
    return ldg_chk(a.q + (int64_t)c * a.q_stride) *
           (a.g ? ldg_chk(a.g + (int64_t)c * a.g_stride) : 1.0f);
}

template <typename T>
__global__ void route_fwd_generic_kernel(const __grid_constant__ RouteArgs a, int wpb)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(16) float gsm[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, r = a.r, H = a.H, N = a.n_src;
    const int K = d / H, Kr = r / H, kstart = d - r;
    const int64_t TT = a.T;
    float *qg = gsm;                                            // [r]
    float *wz = gsm + r + (size_t)warp * gen_fwd_warp_floats(N, H);
    float *lse_s = wz + (size_t)N * H;
    float *cinv = lse_s + H;
    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    for (int c = threadIdx.x; c < r; c += blockDim.x) qg[c] = gen_qg(a, c);
    __syncthreads();
    const T *bank = static_cast<const T *>(a.bank);
    const float alpha = a.alpha ? ldg_chk(a.alpha) : 1.0f;

    for (int64_t t = (int64_t)blockIdx.x * wpb + warp; t < TT; t += (int64_t)gridDim.x * wpb) {
        for (int n = lane; n < N; n += 32) cinv[n] = ldg_chk(a.inv + t * a.inv_ld + s_rows[n]);
        __syncwarp();
        // scores, one warp reduction per (row, head)
        for (int n = 0; n < N; ++n) {
            const T *key = bank + ((int64_t)s_rows[n] * TT + t) * d + kstart;
            for (int h = 0; h < H; ++h) {
                float p = 0.f;
                for (int k = lane; k < Kr; k += 32) p = fmaf(qg[h * Kr + k], gen_ld(key + h * Kr + k), p);
                p = warp_sum(p);
                float z = __fmul_rn(p, cinv[n]);
                if (a.has_bias) z = __fadd_rn(z, a.bias[n]);
                if (lane == 0) wz[n * H + h] = z;
            }
        }
        __syncwarp();
        // softmax per head: lse, then the weights exp(z - lse) in place
        for (int h = lane; h < H; h += 32) {
            float m = wz[h];
            for (int n = 1; n < N; ++n) m = fmaxf(m, wz[n * H + h]);
            float l = 0.f;
            for (int n = 0; n < N; ++n) l += exp2f((wz[n * H + h] - m) * kLog2e);
            const float lse = m + log2f(l) * kLn2;
            lse_s[h] = lse;
            st_chk(a.lse + (t * H + h), lse);
            for (int n = 0; n < N; ++n) wz[n * H + h] = exp2f((wz[n * H + h] - lse) * kLog2e);
        }
        __syncwarp();
        // mix, rows inner
        const int64_t orow = t * d;
        for (int c = lane; c < d; c += 32) {
            const int h = c / K;
            float o = 0.f;
            for (int n = 0; n < N; ++n)
                o = fmaf(wz[n * H + h], gen_ld(bank + ((int64_t)s_rows[n] * TT + t) * d + c), o);
            if (a.routed) st_elem(static_cast<T *>(a.routed) + orow + c, o);
            if (a.partial)
                o = fmaf(alpha, o, gen_ld(static_cast<const T *>(a.partial) + orow + c));
            st_elem(static_cast<T *>(a.out) + orow + c, o);
        }
        __syncwarp();
    }
}

template <typename T>
__global__ void route_bwd_generic_kernel(const __grid_constant__ RouteArgs a, int wpb)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(16) float gsm[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, r = a.r, H = a.H, N = a.n_src;
    const int K = d / H, Kr = r / H, kstart = d - r;
    const int64_t TT = a.T;
    float *qg = gsm;                                            // [r]
    float *W = gsm + r + (size_t)warp * gen_bwd_warp_floats(N, H, r);
    float *DZ = W + (size_t)N * H;
    float *S = DZ + (size_t)N * H;
    float *Cn = S + H;
    float *cinv = Cn + N;
    float *U = cinv + N;                                        // [r]
    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    for (int c = threadIdx.x; c < r; c += blockDim.x) qg[c] = gen_qg(a, c);
    for (int c = lane; c < r; c += 32) U[c] = 0.f;
    __syncthreads();
    const T *bank = static_cast<const T *>(a.bank);
    const T *dout = static_cast<const T *>(a.dout);
    const T *fout = static_cast<const T *>(a.fout);
    const float alpha = a.alpha ? ldg_chk(a.alpha) : 1.0f;
    const float inv_w = 1.0f / (float)(a.norm_full ? d : r);
    const int64_t gw = (int64_t)blockIdx.x * wpb + warp;
    const int64_t GW = (int64_t)gridDim.x * wpb;
    float dal = 0.f;

    for (int64_t t = gw; t < TT; t += GW) {
        const int64_t trow = t * d;
        // coupling term per head, S_h = <G_h, out_h> with G = alpha dL/dh
        float raw = 0.f;
        for (int h = 0; h < H; ++h) {
            float sp = 0.f;
            for (int k = lane; k < K; k += 32) {
                const float gv = gen_ld(dout + trow + h * K + k);
                const float ov = gen_ld(fout + trow + h * K + k);
                raw = fmaf(gv, ov, raw);
                sp = fmaf(alpha * gv, ov, sp);
            }
            sp = warp_sum(sp);
            if (lane == 0) S[h] = a.coupling ? ldg_chk(a.coupling + (t * H + h)) : sp;
        }
        if (a.dalpha) dal += warp_sum(raw);
        for (int n = lane; n < N; n += 32) cinv[n] = ldg_chk(a.inv + t * a.inv_ld + s_rows[n]);
        __syncwarp();
        // per row: value dot P, raw score zr, weight, score gradient, C_n
        for (int n = 0; n < N; ++n) {
            const T *src = bank + ((int64_t)s_rows[n] * TT + t) * d;
            const float iv = cinv[n];
            float C = 0.f;
            for (int h = 0; h < H; ++h) {
                float P = 0.f, zr = 0.f;
                for (int k = lane; k < K; k += 32)
                    P = fmaf(alpha * gen_ld(dout + trow + h * K + k), gen_ld(src + h * K + k), P);
                for (int k = lane; k < Kr; k += 32)
                    zr = fmaf(qg[h * Kr + k], gen_ld(src + kstart + h * Kr + k), zr);
                P = warp_sum(P);
                zr = warp_sum(zr);
                float z = __fmul_rn(zr, iv);
                if (a.has_bias) z = __fadd_rn(z, a.bias[n]);
                const float lse = ldg_chk(a.lse + t * H + h);
                const float w = exp2f((z - lse) * kLog2e);
                const float dz = w * (P - S[h]);
                C = fmaf(dz, zr, C);
                if (lane == 0) {
                    W[n * H + h] = w;
                    DZ[n * H + h] = dz;
                }
            }
            if (lane == 0) Cn[n] = C;
        }
        __syncwarp();
        // gradient rows, rows inner; dq/dg partials on the key coordinates
        for (int c = lane; c < d; c += 32) {
            const int hv = c / K;
            const int kc = c - kstart;
            const bool key = kc >= 0;
            const int hk = key ? kc / Kr : 0;
            const bool norm = a.norm_full || key;
            const float Gc = alpha * gen_ld(dout + trow + c);
            const float qgc = key ? qg[kc] : 0.f;
            float u = key ? U[kc] : 0.f;
            for (int n = 0; n < N; ++n) {
                const int64_t off = ((int64_t)s_rows[n] * TT + t) * d + c;
                const float sv = gen_ld(bank + off);
                const bool first = (a.first_mask[n >> 5] >> (n & 31)) & 1u;
                float v = first ? 0.f : ld_chk(a.grad + off);
                v = fmaf(W[n * H + hv], Gc, v);
                const float iv = cinv[n];
                if (key) {
                    const float ak = iv * DZ[n * H + hk];
                    v = fmaf(ak, qgc, v);
                    u = fmaf(ak, sv, u);
                }
                if (norm) v = fmaf(-(iv * iv * iv * Cn[n] * inv_w), sv, v);
                st_chk(a.grad + off, v);
            }
            if (key) U[kc] = u;
        }
        __syncwarp();
    }
    // the block's dq/dg partial sums (its warps in order) -> workspace row
    // blockIdx.x; dL/dalpha -> tail
    __syncthreads();
    const size_t wf = gen_bwd_warp_floats(N, H, r);
    const float *U0 = gsm + r + (U - W);                        // warp 0's U
    for (int c = threadIdx.x; c < r; c += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < wpb; ++w) s += U0[(size_t)w * wf + c];
        st_chk(a.ws + ((int64_t)blockIdx.x * r + c), s);
    }
    if (a.dalpha) {
        __shared__ float s_dal[4];
        if (lane == 0) s_dal[warp] = dal;
        __syncthreads();
        if (threadIdx.x == 0) {
            float s = 0.f;
            for (int w = 0; w < wpb; ++w) s += s_dal[w];
            float *tail = a.ws + (int64_t)gridDim.x * r + (int64_t)blockIdx.x * 4;
            st_chk(tail, s);   // scalar stores: r may be odd, so the tail may not be 16-byte aligned
            st_chk(tail + 1, 0.f);
            st_chk(tail + 2, 0.f);
            st_chk(tail + 3, 0.f);
        }
    }
}

// The exact coupling term of a site's backward, summed over the sources as in
// the first sweep of "Multi-Head Attention Residuals", Appendix E (Figure 10):
//   S[t, h] = alpha * sum_n w_{n,h} <dL/dout_[h], s_{n,[h]}>,  w = exp(z - lse)
// with the scores recomputed as the forward takes them (z = inv * <q g, key
// slice h>, plus log k for a row listed k times) and alpha the delta form's
// gate (1 otherwise). Every shape: one warp per token, the heads in turn,
// the rows inner, scalar element accesses. The backward kernels read S
// instead of <G_h, out_h> from the stored forward output, whose rounding
// (bf16) would otherwise enter every routing feedback.
template <typename T>
__global__ void route_coupling_kernel(const __grid_constant__ RouteArgs a, float *S_out, int wpb)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(16) float gsm[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, r = a.r, H = a.H, N = a.n_src;
    const int K = d / H, Kr = r / H, kstart = d - r;
    const int64_t TT = a.T;
    float *qg = gsm;                                            // [r]
    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    for (int c = threadIdx.x; c < r; c += blockDim.x) qg[c] = gen_qg(a, c);
    __syncthreads();
    const T *bank = static_cast<const T *>(a.bank);
    const T *dout = static_cast<const T *>(a.dout);
    const float alpha = a.alpha ? ldg_chk(a.alpha) : 1.0f;
    const int64_t gw = (int64_t)blockIdx.x * wpb + warp;
    const int64_t GW = (int64_t)gridDim.x * wpb;
    for (int64_t t = gw; t < TT; t += GW) {
        const int64_t trow = t * d;
        for (int h = 0; h < H; ++h) {
            const float lse = ldg_chk(a.lse + (t * H + h));
            float S = 0.f;
            for (int n = 0; n < N; ++n) {
                const T *src = bank + ((int64_t)s_rows[n] * TT + t) * d;
                float P = 0.f, zr = 0.f;
                for (int k = lane; k < K; k += 32)
                    P = fmaf(gen_ld(dout + trow + h * K + k), gen_ld(src + h * K + k), P);
                for (int k = lane; k < Kr; k += 32)
                    zr = fmaf(qg[h * Kr + k], gen_ld(src + kstart + h * Kr + k), zr);
                P = warp_sum(P);
                zr = warp_sum(zr);
                float z = __fmul_rn(zr, ldg_chk(a.inv + (t * a.inv_ld + s_rows[n])));
                if (a.has_bias) z = __fadd_rn(z, a.bias[n]);
                S = fmaf(exp2f((z - lse) * kLog2e), P, S);
            }
            if (lane == 0) st_chk(S_out + (t * H + h), alpha * S);
        }
    }
}

template <typename T>
cudaError_t dispatch_coupling(const RouteArgs &a, float *S, cudaStream_t s)
{
    constexpr int wpb = 4;
    const size_t smem = (size_t)a.r * 4;
    const void *k = reinterpret_cast<const void *>(&route_coupling_kernel<T>);
    int grid = 0;
    cudaError_t e = persistent_grid(k, wpb * 32, smem, &grid);
    if (e != cudaSuccess) return e;
    const int64_t need = (a.T + wpb - 1) / wpb;
    if (need < grid) grid = (int)need;
    route_coupling_kernel<T><<<grid, wpb * 32, smem, s>>>(a, S, wpb);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_generic_fwd(const RouteArgs &a, cudaStream_t s)
{
    const int wpb = gen_block_warps(gen_fwd_warp_floats(a.n_src, a.H), a.r);
    if (wpb == 0) return cudaErrorNotSupported;
    const size_t smem = ((size_t)a.r + wpb * gen_fwd_warp_floats(a.n_src, a.H)) * 4;
    const void *k = reinterpret_cast<const void *>(&route_fwd_generic_kernel<T>);
    int grid = 0;
    cudaError_t e = persistent_grid(k, wpb * 32, smem, &grid);
    if (e != cudaSuccess) return e;
    const int64_t need = (a.T + wpb - 1) / wpb;
    if (need < grid) grid = (int)need;
    route_fwd_generic_kernel<T><<<grid, wpb * 32, smem, s>>>(a, wpb);
    return cudaGetLastError();
}

// The grid is SMs x kGenBlocksPerSm blocks whatever their warp count, so the
// workspace (one row per block) does not depend on the source count.
template <typename T>
cudaError_t dispatch_generic_bwd(const RouteArgs *a, cudaStream_t s, int *grid_rows)
{
    int blocks = 0;
    cudaError_t e = generic_bwd_rows(&blocks);
    if (e != cudaSuccess) return e;
    if (grid_rows) {
        *grid_rows = blocks;
        return cudaSuccess;
    }
    const int wpb = gen_block_warps(gen_bwd_warp_floats(a->n_src, a->H, a->r), a->r);
    if (wpb == 0) return cudaErrorNotSupported;
    const size_t smem = ((size_t)a->r + wpb * gen_bwd_warp_floats(a->n_src, a->H, a->r)) * 4;
    const void *k = reinterpret_cast<const void *>(&route_bwd_generic_kernel<T>);
    int unused = 0;
    e = persistent_grid(k, wpb * 32, smem, &unused);  // shared-memory opt-in
    if (e != cudaSuccess) return e;
    route_bwd_generic_kernel<T><<<blocks, wpb * 32, smem, s>>>(*a, wpb);
    return cudaGetLastError();
}

}  // namespace ar

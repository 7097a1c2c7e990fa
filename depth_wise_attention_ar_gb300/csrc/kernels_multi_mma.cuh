// Multi-query forward for bf16 rows with the two per-token contractions on
// tensor cores (warp-level mma.sync m16n8k16, fp32 accumulation).
//
// Same result as the CUDA-core kernel in kernels_multi.cuh (the reads of nq
// sites over one row list, "Low-Rank Attention Residuals", Sec. 3.4), for up
// to 16 rows and 8 queries. Per token, with the token's N rows staged in
// shared memory (bf16, one bulk copy per row, two token buffers):
//   scores  Z_h[n][i] = sum_{c in key slice h} K[n][c] (q_i g_i)[c]
//           A = rows (16 x 16 tiles, rows past N read a zero line),
//           B = q_i g_i as two bf16 parts (hi + lo = the fp32 value to 16
//           bits), so the scores carry fp32-like precision;
//   softmax per (query, head) over the rows, in fp32: weights and lse;
//   mix     out_i[c] = sum_n P_h[i][n] V[n][c]
//           A = weights (hi + lo bf16 parts, rows past nq and columns past N
//           zero), B = 8-column tiles of the staged rows (ldmatrix.trans).
// This is a dense contraction per token, but with M = 8 queries and K <= 16
// rows: far below the 64-row minimum of the sm_100 tcgen05 MMA, so the
// warp-level MMA is the fitting unit; the kernel stays bound by HBM.
#pragma once

#include "common.cuh"
#include "launch_util.cuh"

namespace ar {

constexpr int kMmaThreads = 256;      // 8 warps
constexpr int kMmaMaxRows = 16;
// per-warp output staging: 8 query rows of 64 bf16 columns, rows 144 bytes
// apart (conflict-free 4-byte writes and 16-byte reads)
constexpr int kStgPitch = 144;
// key-slice steps of 16 columns held in registers: key slices up to 256 wide
constexpr int kMmaMaxSteps = 16;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t r[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// c += a (16x16, row-major) * b (16x8, column-major), bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two adjacent 8-column output tiles (the second only if `two`): head h's
// weight fragments are (re)loaded when the head changes, the four MMAs
// (weights hi + lo, two tiles) are issued before any result is used, and the
// query rows go to the warp's staging buffer at tile slots slot, slot + 1.
__device__ __forceinline__ void mix_pair(int tile, int slot, bool two, int K, int H, int lane,
                                         const __nv_bfloat16 *pw, const uint32_t (&bq)[4],
                                         int &hcur, uint32_t (&ah)[4], uint32_t (&al)[4],
                                         unsigned char *stg)
{
    auto load_head = [&](int h) {  // weights of head h: A rows = queries, columns = rows n
        const uint32_t aoff = ((h * 16 + (lane & 15)) * 16 + ((lane >> 4) << 3)) * 2;
        ldsm_x4(smem_u32(pw) + aoff, ah);
        ldsm_x4(smem_u32(pw + (size_t)H * 256) + aoff, al);
        hcur = h;
    };
    const int h0 = tile * 8 / K, h1 = (tile + 1) * 8 / K;
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    if (h0 != hcur) load_head(h0);
    mma_16816(c0, ah, bq[0], bq[1]);
    mma_16816(d0, al, bq[0], bq[1]);
    if (two) {
        if (h1 != hcur) load_head(h1);
        mma_16816(c1, ah, bq[2], bq[3]);
        mma_16816(d1, al, bq[2], bq[3]);
    }
    // row = query lane / 4, columns 2 (lane % 4), + 1 of each tile
    unsigned char *row = stg + (lane >> 2) * kStgPitch + 4 * (lane & 3);
    *reinterpret_cast<__nv_bfloat162 *>(row + slot * 16) =
        __floats2bfloat162_rn(c0[0] + d0[0], c0[1] + d0[1]);
    if (two)
        *reinterpret_cast<__nv_bfloat162 *>(row + (slot + 1) * 16) =
            __floats2bfloat162_rn(c1[0] + d1[0], c1[1] + d1[1]);
}

inline size_t multi_mma_fixed_bytes(int r, int H)
{
    return 2 * 8                                   // mbarriers
           + 16                                    // a zero line
           + (size_t)AR_MAX_QUERIES * H * 16 * 4   // scores [8][H][16]
           + 2 * (size_t)H * 16 * 16 * 2           // weights, hi and lo [2][H][16][16]
           + (size_t)kMmaMaxRows * 4               // inverse RMS
           + (size_t)(kMmaThreads / 32) * 8 * kStgPitch;  // output staging
}

// Token buffers per block, with the shared-memory size: one when two blocks
// then share an SM (each covers the other's loads), else two when they fit,
// else one; 0 when none fits.
inline int multi_mma_buffers(int d, int r, int H, int N, size_t *smem)
{
    const size_t fixed = multi_mma_fixed_bytes(r, H);
    const size_t tok = (size_t)N * (d * 2 + 16);
    if (2 * (tok + fixed + 1024) <= 228 * 1024) {
        *smem = tok + fixed;
        return 1;
    }
    for (int nb = 2; nb >= 1; --nb)
        if (nb * tok + fixed <= 200 * 1024) {
            *smem = nb * tok + fixed;
            return nb;
        }
    return 0;
}

__global__ void __launch_bounds__(kMmaThreads)
    route_fwd_multi_mma_kernel(const __grid_constant__ MultiArgs m, int nbuf)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[kMmaMaxRows];
    constexpr int QM = AR_MAX_QUERIES;
    const RouteArgs &a = m.base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int d = a.d, r = a.r, N = a.n_src, H = a.H, nq = m.nq;
    const int64_t TT = a.T;
    // staged rows are padded by 16 bytes, so the 8 row addresses of an
    // ldmatrix fall on different shared-memory banks
    const uint32_t row_bytes = (uint32_t)d * 2u, pitch = row_bytes + 16u;
    const uint32_t tok_bytes = (uint32_t)N * row_bytes, tok_pitch = (uint32_t)N * pitch;
    const int K = d / H, Kr = r / H, kcol0 = d - r;

    if (tid < N) s_rows[tid] = a.rows[tid];
    unsigned char *bufs = smem;
    unsigned char *p = bufs + (size_t)nbuf * tok_pitch;
    uint64_t *bars = reinterpret_cast<uint64_t *>(p);
    p += 16;
    unsigned char *zline = p;                                   // 16 zero bytes
    p += 16;
    float *zs = reinterpret_cast<float *>(p);                   // [8][H][16]
    p += (size_t)QM * H * 16 * 4;
    __nv_bfloat16 *pw = reinterpret_cast<__nv_bfloat16 *>(p);   // [2][H][16][16]
    p += 2 * (size_t)H * 16 * 16 * 2;
    float *invs = reinterpret_cast<float *>(p);                 // [16]
    p += (size_t)kMmaMaxRows * 4;
    unsigned char *stg = p + (size_t)warp * 8 * kStgPitch;      // this warp's staging

    // B fragments of q*g for this warp's head (warp h < H), in two bf16 parts:
    // b0 = (key columns 2 t4, 2 t4 + 1; query g8), b1 = the same 8 columns on,
    // per 16-column step of the key slice; queries past nq are zero
    const int nks = Kr / 16;
    uint32_t qh[kMmaMaxSteps][2], ql[kMmaMaxSteps][2];
#pragma unroll
    for (int ks = 0; ks < kMmaMaxSteps; ++ks)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float v[2] = {0.f, 0.f};
            if (warp < H && ks < nks && g8 < nq) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = warp * Kr + ks * 16 + half * 8 + 2 * t4 + e;
                    v[e] = __ldg(m.q[g8] + c) * (m.g[g8] ? __ldg(m.g[g8] + c) : 1.0f);
                }
            }
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v[0], v[1]);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0] - __low2float(hi), v[1] - __high2float(hi));
            qh[ks][half] = *reinterpret_cast<const uint32_t *>(&hi);
            ql[ks][half] = *reinterpret_cast<const uint32_t *>(&lo);
        }
    // zero weights and zero line
    for (int i = tid; i < 2 * H * 256; i += kMmaThreads) pw[i] = __float2bfloat16_rn(0.f);
    if (tid < 4) reinterpret_cast<uint32_t *>(zline)[tid] = 0u;
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t GB = gridDim.x, gb = blockIdx.x;
    const uint64_t pol = l2_policy_evict_first();
    auto issue_token = [&](int64_t tok, int b) {  // thread 0: all N rows of a token
        unsigned char *dst = bufs + (size_t)b * tok_pitch;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[b], tok_bytes);
        for (int n = 0; n < N; ++n)
            bulk_g2s(dst + (size_t)n * pitch,
                     static_cast<const unsigned char *>(a.bank) +
                         ((int64_t)s_rows[n] * TT + tok) * row_bytes,
                     row_bytes, &bars[b], pol);
    };
    if (tid == 0)
        for (int b = 0; b < nbuf; ++b)
            if (gb + b * GB < TT) issue_token(gb + b * GB, b);

    const uint32_t zaddr = smem_u32(zline);
    const int ntile = d / 8, ngroups = (ntile + 7) / 8;
    uint32_t phase = 0;
    int b = 0;
    bool ok = true;
    for (int64_t tok = gb; tok < TT; tok += GB) {
        if (tid < N) invs[tid] = __ldg(a.inv + tok * a.inv_ld + s_rows[tid]);
        const bool got = mbar_wait(&bars[b], (phase >> b) & 1u, kWaitLimit);
        if (__syncthreads_or(!got)) { ok = false; break; }
        phase ^= 1u << b;
        const uint32_t buf = smem_u32(bufs + (size_t)b * tok_pitch);

        // 1. scores on tensor cores: warp h computes head h
        if (warp < H) {
            const int h = warp;
            float c[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
            const int rowA = lane & 15;
#pragma unroll
            for (int ks = 0; ks < kMmaMaxSteps; ++ks) {
                if (ks >= nks) break;
                const int col = kcol0 + h * Kr + ks * 16 + ((lane >> 4) << 3);
                uint32_t af[4];
                ldsm_x4(rowA < N ? buf + rowA * pitch + col * 2 : zaddr, af);
                mma_16816(c, af, qh[ks][0], qh[ks][1]);    // two chains: hi and lo parts
                mma_16816(cl, af, ql[ks][0], ql[ks][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) c[e] += cl[e];
            // c0, c1: row n = g8, queries 2 t4, 2 t4 + 1; c2, c3: row n = g8 + 8
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = g8 + ((e >> 1) << 3), qi = 2 * t4 + (e & 1);
                if (n < N && qi < nq) {
                    float z = __fmul_rn(c[e], invs[n]);
                    if (a.has_bias) z = __fadd_rn(z, a.bias[n]);
                    zs[(qi * H + h) * 16 + n] = z;
                }
            }
        }
        __syncthreads();

        // 2. weights (hi + lo bf16 parts) and lse per (query, head), fp32
        if (tid < nq * H) {
            const int qi = tid / H, hh = tid - qi * H;
            const float *zq = zs + (qi * H + hh) * 16;
            float mx = zq[0];
            for (int n = 1; n < N; ++n) mx = fmaxf(mx, zq[n]);
            float l = 0.f;
            for (int n = 0; n < N; ++n) l += exp2f((zq[n] - mx) * kLog2e);
            const float lse = mx + log2f(l) * kLn2;
            __nv_bfloat16 *wh = pw + ((size_t)hh * 16 + qi) * 16;
            __nv_bfloat16 *wl = wh + (size_t)H * 256;
            for (int n = 0; n < N; ++n) {
                const float w = exp2f((zq[n] - lse) * kLog2e);
                const __nv_bfloat16 hi = __float2bfloat16_rn(w);
                wh[n] = hi;
                wl[n] = __float2bfloat16_rn(w - __bfloat162float(hi));
            }
            m.lse[qi][tok * H + hh] = lse;
        }
        __syncthreads();

        // 3. mix on tensor cores, per warp in groups of 64 columns (8 tiles of
        // 8): two tiles per ldmatrix, the outputs staged in the warp's buffer
        // and written as 16-byte row pieces (whole 128-byte row segments)
        int hcur = -1;
        uint32_t ah[4], al[4];
        for (int gi = warp; gi < ngroups; gi += kMmaThreads / 32) {
            const int t0 = gi * 8;
            for (int tp = 0; tp < 8 && t0 + tp < ntile; tp += 2) {
                const int ta = t0 + tp;
                const bool two = ta + 1 < ntile;
                const int kr = lane & 15, tl = ta + (two ? (lane >> 4) : 0);
                uint32_t bq[4];
                ldsm_x4_trans(kr < N ? buf + kr * pitch + tl * 16 : zaddr, bq);
                mix_pair(ta, tp, two, K, H, lane, pw, bq, hcur, ah, al, stg);
            }
            __syncwarp();
            for (int idx = lane; idx < 64; idx += 32) {
                const int row = idx >> 3, seg = idx & 7;
                if (row < nq && t0 + seg < ntile)
                    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(m.out[row]) + tok * d +
                                               (t0 + seg) * 8) =
                        *reinterpret_cast<const uint4 *>(stg + row * kStgPitch + seg * 16);
            }
            __syncwarp();
        }
        // every thread is done with this buffer: the token nbuf steps ahead
        // can land in it
        __syncthreads();
        if (tid == 0 && tok + nbuf * GB < TT) issue_token(tok + nbuf * GB, b);
        if (++b == nbuf) b = 0;
    }
    if (!ok && tid == 0) {
        report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
        for (int k = 0; k < nbuf; ++k) {
            mbar_wait(&bars[b], (phase >> b) & 1u, 1u << 16);
            phase ^= 1u << b;
            if (++b == nbuf) b = 0;
        }
    }
}

// bf16 rows, at most 16 rows, at most 8 heads (a warp per head for the
// scores), key slices of whole 16-column steps up to 256 columns, 8-column
// tiles within a head. Returns cudaErrorNotSupported otherwise. (This header
// belongs to one translation unit: the definition below is not inline.)
cudaError_t dispatch_fwd_multi_mma(const MultiArgs &m, cudaStream_t s)
{
    const RouteArgs &a = m.base;
    if (a.n_src > kMmaMaxRows || (a.r / a.H) % 16 != 0 || a.r / a.H > 16 * kMmaMaxSteps ||
        (a.d / a.H) % 8 != 0 || a.d % 8 != 0 || a.H > kMmaThreads / 32)
        return cudaErrorNotSupported;
    size_t smem = 0;
    const int nbuf = multi_mma_buffers(a.d, a.r, a.H, a.n_src, &smem);
    if (nbuf == 0) return cudaErrorNotSupported;
    const void *k = reinterpret_cast<const void *>(&route_fwd_multi_mma_kernel);
    int grid = 0;
    cudaError_t e = persistent_grid(k, kMmaThreads, smem, &grid);
    if (e != cudaSuccess) return e;
    if (a.T < grid) grid = (int)a.T;
    route_fwd_multi_mma_kernel<<<grid, kMmaThreads, smem, s>>>(m, nbuf);
    return cudaGetLastError();
}

}  // namespace ar

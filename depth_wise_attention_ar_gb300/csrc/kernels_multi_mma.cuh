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

inline size_t multi_mma_fixed_bytes(int H)
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
    const size_t fixed = multi_mma_fixed_bytes(H);
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
    AR_CHK_ENTER(m.base);
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
                    v[e] = ldg_chk(m.q[g8] + c) * (m.g[g8] ? ldg_chk(m.g[g8] + c) : 1.0f);
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
        if (tid < N) invs[tid] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[tid]);
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
            st_chk(m.lse[qi] + (tok * H + hh), lse);
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
                    st16_chk(static_cast<__nv_bfloat16 *>(m.out[row]) + tok * d + (t0 + seg) * 8,
                             *reinterpret_cast<const uint4 *>(stg + row * kStgPitch + seg * 16));
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
            mbar_wait(&bars[b], (phase >> b) & 1u, kDrainLimit);
            phase ^= 1u << b;
            if (++b == nbuf) b = 0;
        }
    }
}

// ---- column-tiled streaming version -----------------------------------------
// One block per SM: 8 consumer warps and one producer warp. A token's rows go
// through a ring of S column tiles (all N rows x TC columns, one bulk copy
// per row): first the tiles that hold the key tail (the scores need them),
// then the others, token after token, so the next token's tiles land while
// this token's are mixed. full[s] completes when tile s has landed; each
// consumer warp arrives on empty[s] once it has mixed its part of tile s, and
// the producer refills s after all eight have.
constexpr int kMsWarps = 8;                       // consumer warps
constexpr int kMsThreads = (kMsWarps + 1) * 32;   // + the producer warp
constexpr int kMsMaxStages = 16;
constexpr int kMsZp = 20;   // score row pitch (floats): conflict-free softmax reads

struct MsLayout {
    int TC, tc_shift, ntiles, kt0, nk, S;   // tile width (2^tc_shift), tiles per row,
                                            // first key tile, key tiles, ring
    uint32_t row_pitch, tile_pitch, qg_pitch;
    size_t smem;
};

// The ring must hold a token's key tiles plus at least one more tile.
inline bool ms_layout(int d, int r, int H, int N, MsLayout *L)
{
    L->TC = d % 512 == 0 ? 512 : 256;
    L->tc_shift = L->TC == 512 ? 9 : 8;
    if (d % L->TC != 0) return false;
    L->ntiles = d / L->TC;
    L->kt0 = (d - r) / L->TC;
    L->nk = L->ntiles - L->kt0;
    L->row_pitch = (uint32_t)L->TC * 2u + 16u;   // 16-byte pad: conflict-free ldmatrix rows
    L->tile_pitch = (uint32_t)N * L->row_pitch;
    L->qg_pitch = (uint32_t)r * 2u + 16u;
    const size_t fixed = 2 * (size_t)kMsMaxStages * 8 + 16 + (size_t)AR_MAX_QUERIES * H * kMsZp * 4 +
                         2 * (size_t)H * 256 * 2 + 2 * (size_t)kMmaMaxRows * 4 +
                         (size_t)kMsWarps * 8 * kStgPitch + 2 * (size_t)AR_MAX_QUERIES * L->qg_pitch;
    // two blocks per SM when a ring deeper than the key tiles fits in half
    // the shared memory, else one
    for (const size_t budget : {(size_t)112 * 1024, (size_t)200 * 1024})
        for (int S = kMsMaxStages; S > L->nk; --S)
            if ((size_t)S * L->tile_pitch + fixed <= budget) {
                L->S = S;
                L->smem = (size_t)S * L->tile_pitch + fixed;
                return true;
            }
    return false;
}

__device__ __forceinline__ void ms_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kMsWarps * 32) : "memory");
}
// Named barrier over the consumer warps that also ORs a flag across them.
__device__ __forceinline__ bool ms_bar_or(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kMsWarps * 32)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kMsThreads, 2)
    route_fwd_multi_stream_kernel(const __grid_constant__ MultiArgs m, const MsLayout L)
{
    AR_CHK_ENTER(m.base);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[kMmaMaxRows];
    __shared__ volatile int s_abort;
    constexpr int QM = AR_MAX_QUERIES;
    constexpr unsigned FULL = 0xffffffffu;
    const RouteArgs &a = m.base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int d = a.d, r = a.r, N = a.n_src, H = a.H, nq = m.nq;
    const int64_t TT = a.T;
    const int K = d / H, Kr = r / H, kcol0 = d - r;
    const int TC = L.TC, ntiles = L.ntiles, kt0 = L.kt0, nk = L.nk, S = L.S;
    const uint32_t rp = L.row_pitch, tp = L.tile_pitch;

    if (tid < N) s_rows[tid] = a.rows[tid];
    if (tid == 0) s_abort = 0;
    unsigned char *ring = smem;
    unsigned char *p = ring + (size_t)S * tp;
    uint64_t *full = reinterpret_cast<uint64_t *>(p);
    uint64_t *empty = full + kMsMaxStages;
    p += 2 * (size_t)kMsMaxStages * 8;
    unsigned char *zline = p;                                   // 16 zero bytes
    p += 16;
    float *zs = reinterpret_cast<float *>(p);                   // [8][H][kMsZp]
    p += (size_t)QM * H * kMsZp * 4;
    __nv_bfloat16 *pw = reinterpret_cast<__nv_bfloat16 *>(p);   // [2][H][16][16]
    p += 2 * (size_t)H * 16 * 16 * 2;
    float *invs = reinterpret_cast<float *>(p);                 // [2][16]
    p += 2 * (size_t)kMmaMaxRows * 4;
    unsigned char *stg = p + (size_t)(warp < kMsWarps ? warp : 0) * 8 * kStgPitch;
    p += (size_t)kMsWarps * 8 * kStgPitch;
    // q*g of every query over the key columns as bf16 hi and lo parts,
    // [part][query][key column], rows padded: the scores' B operands
    unsigned char *qgs = p;
    const uint32_t qgp = L.qg_pitch;
    for (int i = tid; i < QM * r; i += kMsThreads) {
        const int qi = i / r, c = i - qi * r;
        const float v = qi < nq ? ldg_chk(m.q[qi] + c) * (m.g[qi] ? ldg_chk(m.g[qi] + c) : 1.0f) : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        *reinterpret_cast<__nv_bfloat16 *>(qgs + (size_t)qi * qgp + c * 2) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(qgs + (size_t)(QM + qi) * qgp + c * 2) =
            __float2bfloat16_rn(v - __bfloat162float(hi));
    }

    for (int i = tid; i < 2 * H * 256; i += kMsThreads) pw[i] = __float2bfloat16_rn(0.f);
    if (tid < 4) reinterpret_cast<uint32_t *>(zline)[tid] = 0u;
    if (tid == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kMsWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t GB = gridDim.x, gb = blockIdx.x;
    const int64_t ntok = gb < TT ? (TT - 1 - gb) / GB + 1 : 0;

    if (warp == kMsWarps) {
        // ---- producer warp: tiles in the consumers' order, at most S ahead;
        // lane 0 waits for the slot and arms its barrier, lane n copies row n
        const uint64_t pol = l2_policy_evict_first();
        const uint32_t tbytes = (uint32_t)TC * 2u;
        const unsigned char *bank = static_cast<const unsigned char *>(a.bank);
        const unsigned char *src_row =
            lane < N ? bank + (int64_t)s_rows[lane] * TT * d * 2 : bank;
        int st = 0, round = 0;
        int64_t issued = 0;
        bool stop = false;
        for (int64_t ti = 0; ti < ntok && !stop; ++ti) {
            const unsigned char *src_tok = src_row + (gb + ti * GB) * (int64_t)d * 2;
            for (int k = 0; k < ntiles; ++k) {
                const int tile = kt0 + k < ntiles ? kt0 + k : kt0 + k - ntiles;
                int ok = 1;
                if (lane == 0) {
                    if (round > 0 && !mbar_wait(&empty[st], (uint32_t)((round - 1) & 1), kWaitLimit)) {
                        s_abort = 1;
                        report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
                    }
                    ok = !s_abort;
                    if (ok) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(&full[st], (uint32_t)N * tbytes);
                    }
                }
                ok = __shfl_sync(FULL, ok, 0);
                if (!ok) {
                    stop = true;
                    break;
                }
                if (lane < N)
                    bulk_g2s(ring + (size_t)st * tp + (size_t)lane * rp, src_tok + (int64_t)tile * TC * 2,
                             tbytes, &full[st], pol);
                ++issued;
                if (++st == S) {
                    st = 0;
                    ++round;
                }
            }
        }
        // the copies still in flight (among the last S issued) land before
        // the block can leave
        if (lane == 0) {
            int s2 = st, r2 = round;
            for (int64_t j = 0; j < (issued < S ? issued : S); ++j) {
                if (--s2 < 0) {
                    s2 = S - 1;
                    --r2;
                }
                mbar_wait(&full[s2], (uint32_t)(r2 & 1), kDrainLimit);
            }
        }
        return;
    }

    // ---- consumers
    const int nks = Kr / 16;
    // this lane's two output rows of the staged 64-column pieces
    const int orow0 = lane >> 3, oseg = lane & 7;
    __nv_bfloat16 *out0 = orow0 < nq ? static_cast<__nv_bfloat16 *>(m.out[orow0]) : nullptr;
    __nv_bfloat16 *out1 = orow0 + 4 < nq ? static_cast<__nv_bfloat16 *>(m.out[orow0 + 4]) : nullptr;
    // softmax lanes: four per (query, head) pair, rows n = sub, sub + 4, ...
    const int spair = tid >> 2, ssub = tid & 3;
    const int sq = spair / H, sh = spair - sq * H;
    const bool sact = spair < nq * H;
    float *lse_out = sact ? m.lse[sq] : nullptr;

    const uint32_t zaddr = smem_u32(zline), ring_a = smem_u32(ring), qg_a = smem_u32(qgs);
    const int ntl = TC / 8, ngr = ntl / 8;   // 8-column MMA tiles, groups of 8 per tile
    const bool one_head = K % 64 == 0;       // every 64-column group within one head
    int st0 = 0, rnd0 = 0;                   // ring slot and round of the token's first tile
    bool bad = false;
    for (int64_t ti = 0; ti < ntok; ++ti) {
        const int64_t tok = gb + ti * GB;
        float *inv_t = invs + (ti & 1) * kMmaMaxRows;
        if (tid < N) inv_t[tid] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[tid]);
        bool got = true;
        for (int k = 0; k < nk && got; ++k) {
            int sk = st0 + k, rk = rnd0;
            if (sk >= S) {
                sk -= S;
                ++rk;
            }
            got = mbar_wait(&full[sk], (uint32_t)(rk & 1), kWaitLimit);
        }
        if (ms_bar_or(!got || bad)) {
            bad = true;
            break;
        }

        // 1. scores on tensor cores: warp h computes head h from the key tiles
        if (warp < H) {
            const int h = warp;
            float c[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
            float c2[4] = {0.f, 0.f, 0.f, 0.f}, cl2[4] = {0.f, 0.f, 0.f, 0.f};
            const int rowA = lane & 15;
#pragma unroll
            for (int ks = 0; ks < kMmaMaxSteps; ++ks) {
                if (ks >= nks) break;
                const int col = kcol0 + h * Kr + ks * 16 + ((lane >> 4) << 3);
                const int tile = col >> L.tc_shift;
                int sk = st0 + (tile - kt0);
                if (sk >= S) sk -= S;
                uint32_t af[4], bh0, bh1, bl0, bl1;
                ldsm_x4(rowA < N ? ring_a + sk * tp + rowA * rp + (col & (TC - 1)) * 2 : zaddr, af);
                const uint32_t qa = qg_a + (lane & 7) * qgp +
                                    (h * Kr + ks * 16 + ((lane >> 3) & 1) * 8) * 2;
                ldsm_x2(qa, bh0, bh1);
                ldsm_x2(qa + QM * qgp, bl0, bl1);
                // four accumulation chains: q*g hi and lo parts, even and odd steps
                if (ks & 1) {
                    mma_16816(c2, af, bh0, bh1);
                    mma_16816(cl2, af, bl0, bl1);
                } else {
                    mma_16816(c, af, bh0, bh1);
                    mma_16816(cl, af, bl0, bl1);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) c[e] = (c[e] + c2[e]) + (cl[e] + cl2[e]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = g8 + ((e >> 1) << 3), qi = 2 * t4 + (e & 1);
                if (n < N && qi < nq) {
                    float z = __fmul_rn(c[e], inv_t[n]);
                    if (a.has_bias) z = __fadd_rn(z, a.bias[n]);
                    zs[(qi * H + h) * kMsZp + n] = z;
                }
            }
        }
        ms_bar();

        // 2. weights (hi + lo bf16 parts) and lse per (query, head), fp32;
        // four lanes per pair, combined by shuffles
        {
            const float *zq = zs + (sq * H + sh) * kMsZp;
            float zv[4];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = ssub + 4 * j;
                zv[j] = (sact && n < N) ? zq[n] : -INFINITY;
                mx = fmaxf(mx, zv[j]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
            float l = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (ssub + 4 * j < N) l += exp2f((zv[j] - mx) * kLog2e);
            l += __shfl_xor_sync(FULL, l, 1);
            l += __shfl_xor_sync(FULL, l, 2);
            if (sact) {
                const float lse = mx + log2f(l) * kLn2;
                // head sh's A matrix: rows 0-7 the queries' weights (bf16),
                // rows 8-15 what rounding to bf16 left of them
                __nv_bfloat16 *wh = pw + ((size_t)sh * 16 + sq) * 16;
                __nv_bfloat16 *wl = wh + 8 * 16;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = ssub + 4 * j;
                    if (n < N) {
                        const float w = exp2f((zv[j] - lse) * kLog2e);
                        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
                        wh[n] = hi;
                        wl[n] = __float2bfloat16_rn(w - __bfloat162float(hi));
                    }
                }
                if (ssub == 0) st_chk(lse_out + (tok * H + sh), lse);
            }
        }
        ms_bar();

        // 3. mix every tile of the token in sequence order, then release it
        int hcur = -1;
        uint32_t ah[4];
        int sk = st0, rk = rnd0;
        for (int k = 0; k < ntiles; ++k) {
            if (k >= nk && !bad && !mbar_wait(&full[sk], (uint32_t)(rk & 1), kWaitLimit)) bad = true;
            if (!bad) {
                const int tile = kt0 + k < ntiles ? kt0 + k : kt0 + k - ntiles;
                const uint32_t base = ring_a + sk * tp;
                for (int gi = warp; gi < ngr; gi += kMsWarps) {
                    const int lt0 = gi * 8;
                    const int kr = lane & 15;
                    if (one_head) {
                        // the group's 64 columns lie in one head: its weights
                        // once, four B loads, then eight independent MMAs
                        const int h = (tile * ntl + lt0) * 8 / K;
                        if (h != hcur) {
                            ldsm_x4(smem_u32(pw) + ((h * 16 + (lane & 15)) * 16 + ((lane >> 4) << 3)) * 2,
                                    ah);
                            hcur = h;
                        }
                        uint32_t bq[4][4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ldsm_x4_trans(kr < N ? base + kr * rp + (lt0 + 2 * q + (lane >> 4)) * 16
                                                 : zaddr,
                                          bq[q]);
                        float c[8][4];
#pragma unroll
                        for (int t = 0; t < 8; ++t)
#pragma unroll
                            for (int e = 0; e < 4; ++e) c[t][e] = 0.f;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            mma_16816(c[2 * q], ah, bq[q][0], bq[q][1]);
                            mma_16816(c[2 * q + 1], ah, bq[q][2], bq[q][3]);
                        }
                        // query g8: its bf16 part (c0, c1) plus its remainder (c2, c3)
                        unsigned char *srow = stg + (lane >> 2) * kStgPitch + 4 * (lane & 3);
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            *reinterpret_cast<__nv_bfloat162 *>(srow + t * 16) =
                                __floats2bfloat162_rn(c[t][0] + c[t][2], c[t][1] + c[t][3]);
                    } else {
                        // heads change inside the group: per 8-column tile
#pragma unroll
                        for (int tpair = 0; tpair < 8; tpair += 2) {
                            const int tl = lt0 + tpair + (lane >> 4);
                            uint32_t bq[4];
                            ldsm_x4_trans(kr < N ? base + kr * rp + tl * 16 : zaddr, bq);
                            unsigned char *srow = stg + (lane >> 2) * kStgPitch + 4 * (lane & 3);
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int h = ((tile * ntl + lt0 + tpair + u) * 8) / K;
                                if (h != hcur) {
                                    ldsm_x4(smem_u32(pw) +
                                                ((h * 16 + (lane & 15)) * 16 + ((lane >> 4) << 3)) * 2,
                                            ah);
                                    hcur = h;
                                }
                                float c[4] = {0.f, 0.f, 0.f, 0.f};
                                mma_16816(c, ah, bq[2 * u], bq[2 * u + 1]);
                                *reinterpret_cast<__nv_bfloat162 *>(srow + (tpair + u) * 16) =
                                    __floats2bfloat162_rn(c[0] + c[2], c[1] + c[3]);
                            }
                        }
                    }
                    __syncwarp();
                    const int64_t o = tok * d + (int64_t)(tile * ntl + lt0 + oseg) * 8;
                    if (out0)
                        st16_chk(out0 + o, *reinterpret_cast<const uint4 *>(stg + orow0 * kStgPitch + oseg * 16));
                    if (out1)
                        st16_chk(out1 + o,
                                 *reinterpret_cast<const uint4 *>(stg + (orow0 + 4) * kStgPitch + oseg * 16));
                    __syncwarp();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sk]);
            if (++sk == S) {
                sk = 0;
                ++rk;
            }
        }
        st0 = sk;
        rnd0 = rk;
    }
    if (bad && tid == 0) {
        s_abort = 1;
        report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
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
    MsLayout L;
    if (ms_layout(a.d, a.r, a.H, a.n_src, &L)) {
        const void *k = reinterpret_cast<const void *>(&route_fwd_multi_stream_kernel);
        int grid = 0;
        cudaError_t e = persistent_grid(k, kMsThreads, L.smem, &grid);
        if (e != cudaSuccess) return e;
        if (a.T < grid) grid = (int)a.T;
        route_fwd_multi_stream_kernel<<<grid, kMsThreads, L.smem, s>>>(m, L);
        return cudaGetLastError();
    }
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

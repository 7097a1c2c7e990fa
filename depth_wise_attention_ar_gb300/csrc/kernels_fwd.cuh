// Fused routing forward for sm_103a, full-width keys (r = d).
//
// Computes, for one routing site and every token t, the per-head softmax
// over the listed sources and the mixed output ("Multi-Head Attention
// Residuals", Eq. 3; the fused online-softmax design of its Appendix E,
// Figure 9), with the RMSNorm key taken from the cached inverse RMS.
//
// GB300 mapping
// - One warp owns one token at a time and walks its N source rows. Each row
//   (d elements, contiguous) is brought into a per-warp ring of shared-memory
//   stages by a single 1-D bulk copy (cp.async.bulk, completion on an
//   mbarrier); lane 0 refills a stage as soon as the warp has consumed it, so
//   every warp keeps kFwdStages rows in flight and no warp waits on another.
// - Lane l serves head h = l / (32/H); the head's d/H coordinates are spread
//   over its 32/H lanes in 8-element chunks (CPL = d/256 chunks per lane), so
//   the per-head score is a reduction over 32/H lanes (log2(32/H) shuffles)
//   and the lane's head weight needs no broadcast. Chunk order is rotated by
//   the head index so that the lanes of the two heads that share a
//   quarter-warp hit different shared-memory banks.
// - The accumulator, q*g and the staged row's values (8*CPL floats each)
//   live in registers; a staged row is read from shared memory once.
// - The softmax is online; the running maximum only moves when a score
//   exceeds it by kRescaleTau, so the accumulator is rarely rescaled. Scores
//   stay in natural units (exp2 only inside the exponent) so that the
//   backward's recomputed score matches bit for bit.
// - Grid: persistent, SM count x resident blocks; tokens strided over warps.
//
// Sliced keys (SK = true, r < d or any r with whole 8-column key chunks per
// head): the same single pass, with head h's score taken from key slice h,
// the h-th r/H block of the last r columns ("Low-Rank Attention Residuals",
// Eq. 11-12). Lane l of head h also holds key chunks key0 + h*ckh + sub +
// LPH*j (ckh = r/(8H) chunks per key slice), in the order and with the sums
// of the sliced-key backward, so both compute the same score bits; the value
// chunks are read after the weight is known, so only the accumulator and q*g
// stay in registers. q*g is held for KM key-chunk slots per lane (a quarter,
// a half or all of CPL, whichever first covers the key tail), and these
// instantiations have their own entry, route_fwd_sk_kernel, compiled for the
// resident blocks fwd_min_blocks gives.
//
// FRESH (full keys, rows up to 1024 wide): the site's append is fused in. The
// new row already sits in its slot; at its item the kernel squares the staged
// values it holds, sums them over the token's lanes, and caches the inverse
// RMS before scoring the row (one launch per site instead of two).
#pragma once

#include "common.cuh"
#include "launch_util.cuh"

namespace ar {

constexpr int kFwdWarps = 4;
constexpr int kFwdStages = 4;


// Sliced keys on rows of 2048 columns or more: three stages per warp, so that
// three blocks fit in shared memory (more warps for the same token count).
__host__ __device__ constexpr int fwd_stages(bool sk, int cpl)
{
    return sk && cpl >= 8 ? 3 : kFwdStages;
}

// Resident blocks the sliced-key bf16 instantiations are compiled for: the
// accumulator (8 CPL floats) and q*g of the key chunks (8 KM floats) set the
// register need; four blocks where that stays within 128 registers without
// spilling, else three, and two for the widest key slices. (fp32 rows fill
// shared memory first: no bound.)
constexpr int fwd_min_blocks(bool sk_bf16, int cpl, int km)
{
    return !sk_bf16 ? 1 : (cpl + km <= 8 ? 4 : (cpl + km <= 13 ? 3 : 2));
}

inline size_t fwd_smem_bytes(int d, size_t esize, int stages = kFwdStages)
{
    return (size_t)kFwdWarps * stages * d * esize + (size_t)kFwdWarps * stages * 8 +
           (size_t)kFwdWarps * AR_MAX_SOURCES * 4;
}

template <typename T, int CPL, bool SK, bool FRESH, int KM>
__device__ __forceinline__ void route_fwd_body(const RouteArgs &a)
{
    static_assert(SK || KM == CPL, "full keys: a lane's key chunks are its value chunks");
    // packed fp32 pairs for the score and the mix (same bits): measured faster
    // on full-key rows of 1280 columns and more (1B forward phase 18.54 ->
    // 17.87 ms), slightly slower on 1024 (350M 7.41 -> 7.45 ms)
    constexpr bool kPacked = !SK && CPL >= 5;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    constexpr int S = fwd_stages(SK, CPL);
    constexpr int CB = ChunkBytes<T>::value;
    constexpr unsigned FULL = 0xffffffffu;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, N = a.n_src, H = a.H;
    const int64_t TT = a.T;
    const uint32_t row_bytes = (uint32_t)d * (uint32_t)sizeof(T);

    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    unsigned char *ring = smem + (size_t)warp * S * row_bytes;
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + (size_t)kFwdWarps * S * row_bytes) + warp * S;
    float *cur_inv = reinterpret_cast<float *>(smem + (size_t)kFwdWarps * S * row_bytes +
                                               (size_t)kFwdWarps * S * 8) +
                     warp * AR_MAX_SOURCES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // ---- lane -> head and chunk mapping
    const int LPH = 32 / H;
    const int h = lane / LPH, sub = lane - h * LPH;
    int cidx[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) cidx[j] = chunk_of<CPL>(h, sub, LPH, j);
    // key chunks: the value chunks themselves for full keys; for sliced keys
    // chunks of key slice h (ceil(r / 256) <= KM of them per lane)
    const int key0 = SK ? (d - a.r) / 8 : 0, ckh = SK ? a.r / 8 / H : 0;
    int kidx[KM];
    bool kval[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        kval[j] = !SK || sub + LPH * j < ckh;
        kidx[j] = SK ? key0 + h * ckh + sub + LPH * j : cidx[j];
    }
    // query times norm weight over this lane's key coordinates; on rows of
    // 1280 columns and more loaded after the first copies are issued, so that
    // the copies' latency starts at once (1B forward phase 17.88 -> 17.74 ms;
    // 350M, 1024 columns, 7.37 -> 7.60 ms, so not there)
    constexpr bool kQgLate = kPacked;
    float qg[KM][8];
    auto load_qg = [&]() {
#pragma unroll
        for (int j = 0; j < KM; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int c = kidx[j] * 8 + e - key0 * 8;
                qg[j][e] = kval[j] ? ldg_chk(a.q + c * a.q_stride) *
                                         (a.g ? ldg_chk(a.g + c * a.g_stride) : 1.0f)
                                   : 0.f;
            }
    };
    if constexpr (!kQgLate) load_qg();

    // ---- work: tokens gw, gw + GW, ...
    const int64_t GW = (int64_t)gridDim.x * kFwdWarps;
    const int64_t gw = (int64_t)blockIdx.x * kFwdWarps + warp;
    const int64_t ntok = gw < TT ? (TT - 1 - gw) / GW + 1 : 0;
    const int64_t total = ntok * N;
    const uint64_t pol = l2_policy_evict_first();

    // producer cursor (all lanes track it; lane 0 issues)
    int64_t issued = 0, tok_p = gw;
    int n_p = 0, slot_p = 0;
    auto issue_next = [&]() {
        if (lane == 0) {
            const unsigned char *src = static_cast<const unsigned char *>(a.bank) +
                                       ((int64_t)s_rows[n_p] * TT + tok_p) * row_bytes;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[slot_p], row_bytes);
            if (!a.lost_copies)
                bulk_g2s(ring + (size_t)slot_p * row_bytes, src, row_bytes, &bars[slot_p], pol);
        }
        ++issued;
        if (++n_p == N) { n_p = 0; tok_p += GW; }
        if (++slot_p == S) slot_p = 0;
    };
    for (int s = 0; s < S && issued < total; ++s) issue_next();
    if constexpr (kQgLate) load_qg();
    const uint32_t wait_limit = a.wait_limit ? a.wait_limit : kWaitLimit;

    // inverse RMS of the next token's sources, prefetched into registers
    float pre_inv[AR_MAX_SOURCES / 32];
    auto prefetch_inv = [&](int64_t tok) {
#pragma unroll
        for (int u = 0; u < AR_MAX_SOURCES / 32; ++u) {
            const int nn = lane + 32 * u;
            if (nn < N) pre_inv[u] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[nn]);
        }
    };
    if (ntok > 0) prefetch_inv(gw);

    int n = 0, slot = 0;
    uint32_t phase = 0;
    int64_t tok = gw, i = 0;
    float m = 0.f, l = 0.f;
    float acc[CPL][8];
    bool ok = true;
    for (; i < total; ++i) {
        if (n == 0) {
#pragma unroll
            for (int u = 0; u < AR_MAX_SOURCES / 32; ++u) {
                const int nn = lane + 32 * u;
                if (nn < N) cur_inv[nn] = pre_inv[u];
            }
            __syncwarp();
            if (tok + GW < TT) prefetch_inv(tok + GW);
        }
        const bool got = mbar_wait(&bars[slot], (phase >> slot) & 1u, wait_limit);
        if (!__all_sync(FULL, got)) { ok = false; break; }
        phase ^= 1u << slot;
        const unsigned char *buf = ring + (size_t)slot * row_bytes;

        // score of this lane's head: q_h . (g * s_n)_[h], times inv_n
        float v[SK ? 1 : CPL][8];
        float zr = 0.f;
        if constexpr (SK) {
#pragma unroll
            for (int j = 0; j < KM; ++j) {
                if (kval[j]) {
                    float kv[8];
                    ld_chunk_s(reinterpret_cast<const T *>(buf + kidx[j] * CB), kv);
                    zr = __fadd_rn(zr, dot8(qg[j], kv));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                ld_chunk_s(reinterpret_cast<const T *>(buf + cidx[j] * CB), v[j]);
                zr = __fadd_rn(zr, kPacked ? dot8p(qg[j], v[j]) : dot8(qg[j], v[j]));
            }
        }
        zr = group_sum(zr, LPH);
        float ivn = cur_inv[n];
        if constexpr (FRESH && !SK) {
            if (n + 1 == a.fresh1) {
                // the row appended with this read: its inverse RMS from the
                // staged (stored) values, over all d columns, into the cache
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < CPL; ++j)
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(v[j][e], v[j][e], ss);
                ss = warp_sum(ss);
                ivn = rsqrtf(fmaf(ss, 1.0f / (float)d, a.eps));
                if (lane == 0) st_chk(const_cast<float *>(a.inv) + (tok * a.inv_ld + s_rows[n]), ivn);
            }
        }
        // __fmul_rn keeps the product uncontracted: the backward recomputes
        // the same bits
        const float z = __fmul_rn(zr, ivn);
        if (n == 0) {  // first source of the token: weight exp(0) = 1 below
            m = z;
            l = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
        }
        const bool need = z > m + kRescaleTau;
        if (__any_sync(FULL, need)) {
            const float sc = need ? exp2f((m - z) * kLog2e) : 1.f;
            m = need ? z : m;
            l *= sc;
#pragma unroll
            for (int j = 0; j < CPL; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] *= sc;
        }
        const float p = exp2f((z - m) * kLog2e);
        l += p;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            if constexpr (SK) {
                float vv[8];
                ld_chunk_s(reinterpret_cast<const T *>(buf + cidx[j] * CB), vv);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(p, vv[e], acc[j][e]);
            } else if constexpr (kPacked) {
                axpy8(p, v[j], acc[j]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(p, v[j][e], acc[j][e]);
            }
        }
        __syncwarp();
        if (issued < total) issue_next();  // refill the stage just consumed

        if (n == N - 1) {
            const float rl = 1.f / l;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = acc[j][e] * rl;
                store_output<T>(a, tok * d + cidx[j] * 8, o);
            }
            if (sub == 0) st_chk(a.lse + (tok * H + h), m + log2f(l) * kLn2);
        }
        if (++n == N) { n = 0; tok += GW; }
        if (++slot == S) slot = 0;
    }

    if (!ok) {
        if (lane == 0) report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
        // wait briefly for this warp's copies still in flight, then leave
        const uint32_t drain = a.wait_limit ? a.wait_limit : kDrainLimit;
        for (int64_t j = i; j < issued; ++j) {
            mbar_wait(&bars[slot], (phase >> slot) & 1u, drain);
            phase ^= 1u << slot;
            if (++slot == S) slot = 0;
        }
    }
}

// Full keys: the register count is left to the compiler (one block per SM
// minimum), which keeps three blocks resident on 1280-column rows.
template <typename T, int CPL, bool FRESH = false>
__global__ void __launch_bounds__(kFwdWarps * 32)
    route_fwd_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    route_fwd_body<T, CPL, false, FRESH, CPL>(a);
}

// Sliced keys: compiled for fwd_min_blocks resident blocks.
template <typename T, int CPL, int KM>
__global__ void __launch_bounds__(kFwdWarps * 32, fwd_min_blocks(sizeof(T) == 2, CPL, KM))
    route_fwd_sk_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    route_fwd_body<T, CPL, true, false, KM>(a);
}

// Two tokens per warp, full keys, rows of 256 or 512 columns, H <= 4.
//
// On short rows the per-row cost of the stage wait, the refill and the loop
// bounds the one-token kernel above by instruction issue. Here a warp serves
// two adjacent tokens at once, one per half-warp: a stage is one bulk copy of
// both tokens' rows of a source (adjacent in the bank). CPL = d / 256 is the
// chunk count of one lane of the one-warp backward; a lane here holds the
// chunks of two backward lanes of its head (sub and sub + LPH, LPH = lanes
// per head here, half the backward's) and keeps their two partial scores
// apart through the in-group butterfly, adding them last: that is the
// backward's reduction tree, so the recomputed score keeps the forward's
// bits. Odd heads take their two backward lanes' chunks in the other order,
// so that the two head groups of a quarter-warp read different bank groups.
template <typename T, int CPL, bool FRESH = false, int NG = AR_MAX_SOURCES / 32, int MINB = 1>
__global__ void __launch_bounds__(kFwdWarps * 32, MINB)
    route_fwd_pair_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    constexpr int S = kFwdStages;
    constexpr int CB = ChunkBytes<T>::value;
    constexpr int NC = 2 * CPL;         // chunks held by one lane
    constexpr unsigned FULL = 0xffffffffu;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, N = a.n_src, H = a.H;
    const int64_t TT = a.T;
    const uint32_t row_bytes = (uint32_t)d * (uint32_t)sizeof(T);
    const uint32_t stage_bytes = 2 * row_bytes;

    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    unsigned char *ring = smem + (size_t)warp * S * stage_bytes;
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + (size_t)kFwdWarps * S * stage_bytes) + warp * S;
    float *inv_warp = reinterpret_cast<float *>(smem + (size_t)kFwdWarps * S * stage_bytes +
                                                (size_t)kFwdWarps * S * 8) +
                      warp * 2 * AR_MAX_SOURCES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // ---- lane -> token of the pair, head and chunks
    const int tt = lane >> 4, fl = lane & 15;
    const int LPHb = 32 / H, LPH = 16 / H;
    const int h = fl / LPH, sub = fl - h * LPH;
    int cidx[NC];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int kk = (k ^ h) & 1;
#pragma unroll
        for (int j = 0; j < CPL; ++j) cidx[k * CPL + j] = chunk_of<CPL>(h, sub + kk * LPH, LPHb, j);
    }
    float qg[NC][8];
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = cidx[j] * 8 + e;
            qg[j][e] = ldg_chk(a.q + c * a.q_stride) * (a.g ? ldg_chk(a.g + c * a.g_stride) : 1.0f);
        }

    // ---- work: token pairs gw, gw + GW, ...
    const int64_t UT = (TT + 1) / 2;
    const int64_t GW = (int64_t)gridDim.x * kFwdWarps;
    const int64_t gw = (int64_t)blockIdx.x * kFwdWarps + warp;
    const int64_t npair = gw < UT ? (UT - 1 - gw) / GW + 1 : 0;
    const int64_t total = npair * N;
    const uint64_t pol = l2_policy_evict_first();

    int64_t issued = 0, u_p = gw;
    int n_p = 0, slot_p = 0;
    auto issue_next = [&]() {
        if (lane == 0) {
            const int64_t t0 = u_p * 2;
            const uint32_t bytes = t0 + 1 < TT ? stage_bytes : row_bytes;  // ragged last pair
            const unsigned char *src = static_cast<const unsigned char *>(a.bank) +
                                       ((int64_t)s_rows[n_p] * TT + t0) * row_bytes;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[slot_p], bytes);
            bulk_g2s(ring + (size_t)slot_p * stage_bytes, src, bytes, &bars[slot_p], pol);
        }
        ++issued;
        if (++n_p == N) { n_p = 0; u_p += GW; }
        if (++slot_p == S) slot_p = 0;
    };
    for (int s = 0; s < S && issued < total; ++s) issue_next();

    // inverse RMS of the next pair's sources, prefetched into registers (NG
    // groups of 32 sources: one group for sites of at most 32 sources)
    float pre_inv[2][NG];
    auto prefetch_inv = [&](int64_t u) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int64_t t = u * 2 + k;
#pragma unroll
            for (int v = 0; v < NG; ++v) {
                const int nn = lane + 32 * v;
                if (nn < N && t < TT) pre_inv[k][v] = ldg_chk(a.inv + t * a.inv_ld + s_rows[nn]);
            }
        }
    };
    if (npair > 0) prefetch_inv(gw);

    int n = 0, slot = 0;
    uint32_t phase = 0;
    int64_t u = gw, i = 0;
    float m = 0.f, l = 0.f;
    float acc[NC][8];
    const float *cur_inv = inv_warp + tt * AR_MAX_SOURCES;
    bool ok = true;
    for (; i < total; ++i) {
        if (n == 0) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int v = 0; v < NG; ++v) {
                    const int nn = lane + 32 * v;
                    if (nn < N) inv_warp[k * AR_MAX_SOURCES + nn] = pre_inv[k][v];
                }
            __syncwarp();
            if (u + GW < UT) prefetch_inv(u + GW);
        }
        const bool got = mbar_wait(&bars[slot], (phase >> slot) & 1u, kWaitLimit);
        if (!__all_sync(FULL, got)) { ok = false; break; }
        phase ^= 1u << slot;
        // this half-warp's token row (the second row of a ragged last pair is
        // stale data: computed on, never stored)
        const unsigned char *buf = ring + (size_t)slot * stage_bytes + (size_t)tt * row_bytes;

        float v[NC][8];
        float z0 = 0.f, z1 = 0.f;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            ld_chunk_s(reinterpret_cast<const T *>(buf + cidx[j] * CB), v[j]);
            if (j < CPL) z0 = __fadd_rn(z0, dot8p(qg[j], v[j]));
            else z1 = __fadd_rn(z1, dot8p(qg[j], v[j]));
        }
        const float zr = __fadd_rn(group_sum(z0, LPH), group_sum(z1, LPH));
        float ivn = cur_inv[n];
        if (FRESH && n + 1 == a.fresh1) {
            // the row appended with this read: its inverse RMS (half-warp sum)
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < NC; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(v[j][e], v[j][e], ss);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
            ivn = rsqrtf(fmaf(ss, 1.0f / (float)d, a.eps));
            const int64_t tk = u * 2 + tt;
            if (fl == 0 && tk < TT)
                st_chk(const_cast<float *>(a.inv) + (tk * a.inv_ld + s_rows[n]), ivn);
        }
        const float z = __fmul_rn(zr, ivn);
        if (n == 0) {
            m = z;
            l = 0.f;
#pragma unroll
            for (int j = 0; j < NC; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
        }
        const bool need = z > m + kRescaleTau;
        if (__any_sync(FULL, need)) {
            const float sc = need ? exp2f((m - z) * kLog2e) : 1.f;
            m = need ? z : m;
            l *= sc;
#pragma unroll
            for (int j = 0; j < NC; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] *= sc;
        }
        const float p = exp2f((z - m) * kLog2e);
        l += p;
#pragma unroll
        for (int j = 0; j < NC; ++j) axpy8(p, v[j], acc[j]);
        __syncwarp();
        if (issued < total) issue_next();

        if (n == N - 1) {
            const int64_t tok = u * 2 + tt;
            if (tok < TT) {
                const float rl = 1.f / l;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = acc[j][e] * rl;
                    store_output<T>(a, tok * d + cidx[j] * 8, o);
                }
                if (sub == 0) st_chk(a.lse + (tok * H + h), m + log2f(l) * kLn2);
            }
        }
        if (++n == N) { n = 0; u += GW; }
        if (++slot == S) slot = 0;
    }

    if (!ok) {
        if (lane == 0) report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
        for (int64_t j = i; j < issued; ++j) {
            mbar_wait(&bars[slot], (phase >> slot) & 1u, kDrainLimit);
            phase ^= 1u << slot;
            if (++slot == S) slot = 0;
        }
    }
}

template <typename T, int CPL, bool FRESH, int NG, int MINB>
cudaError_t launch_fwd_pair_inst(const RouteArgs &a, cudaStream_t s)
{
    const void *k = reinterpret_cast<const void *>(&route_fwd_pair_kernel<T, CPL, FRESH, NG, MINB>);
    const size_t smem = (size_t)kFwdWarps * kFwdStages * 2 * a.d * sizeof(T) +
                        (size_t)kFwdWarps * kFwdStages * 8 +
                        (size_t)kFwdWarps * 2 * AR_MAX_SOURCES * 4;
    int grid = 0;
    cudaError_t e = persistent_grid(k, kFwdWarps * 32, smem, &grid);
    if (e != cudaSuccess) return e;
    route_fwd_pair_kernel<T, CPL, FRESH, NG, MINB><<<grid, kFwdWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

// Sites of at most 32 sources prefetch one inverse RMS per token and lane
// (100M forward phase 1.31 -> 1.23 ms with the suspend hint of the waits; a
// bound of four resident blocks, 128 registers with a small spill, measured
// slower than three).
template <typename T, int CPL, bool FRESH>
cudaError_t launch_fwd_pair_n(const RouteArgs &a, cudaStream_t s)
{
    if (a.n_src <= 32) return launch_fwd_pair_inst<T, CPL, FRESH, 1, 1>(a, s);
    return launch_fwd_pair_inst<T, CPL, FRESH, AR_MAX_SOURCES / 32, 1>(a, s);
}

template <typename T, int CPL>
cudaError_t launch_fwd_pair(const RouteArgs &a, cudaStream_t s)
{
    return a.fresh1 ? launch_fwd_pair_n<T, CPL, true>(a, s) : launch_fwd_pair_n<T, CPL, false>(a, s);
}

template <typename T, int CPL, bool SK, bool FRESH, int KM = CPL>
cudaError_t launch_fwd_inst2(const RouteArgs &a, cudaStream_t s)
{
    const void *k;
    if constexpr (SK)
        k = reinterpret_cast<const void *>(&route_fwd_sk_kernel<T, CPL, KM>);
    else
        k = reinterpret_cast<const void *>(&route_fwd_kernel<T, CPL, FRESH>);
    const size_t smem = fwd_smem_bytes(a.d, sizeof(T), fwd_stages(SK, CPL));
    int grid = 0;
    cudaError_t e = persistent_grid(k, kFwdWarps * 32, smem, &grid);
    if (e != cudaSuccess) return e;
    if constexpr (SK)
        route_fwd_sk_kernel<T, CPL, KM><<<grid, kFwdWarps * 32, smem, s>>>(a);
    else
        route_fwd_kernel<T, CPL, FRESH><<<grid, kFwdWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

// The fresh-row variant only for full keys on rows up to 1024 wide (the host
// sets fresh1 only there: on 1280-wide rows the variant measured slower than
// a separate append).
template <typename T, int CPL, bool SK>
cudaError_t launch_fwd_inst(const RouteArgs &a, cudaStream_t s)
{
    if constexpr (SK) {
        // key chunks per lane: ceil(r / 256), held in the smallest of a
        // quarter, a half or all of the lane's CPL value-chunk slots that fits
        // (q*g of unused slots would otherwise occupy registers)
        constexpr int kQuarter = (CPL + 3) / 4, kHalf = (CPL + 1) / 2;
        const int km = (a.r + 255) / 256;
        if (km <= kQuarter) return launch_fwd_inst2<T, CPL, true, false, kQuarter>(a, s);
        if (km <= kHalf) return launch_fwd_inst2<T, CPL, true, false, kHalf>(a, s);
        return launch_fwd_inst2<T, CPL, true, false, CPL>(a, s);
    } else {
        if constexpr (CPL <= 4) {
            if (a.fresh1) return launch_fwd_inst2<T, CPL, false, true>(a, s);
        }
        return launch_fwd_inst2<T, CPL, false, false>(a, s);
    }
}

// Full-width keys with d = 256 * CPL, CPL in 1..8 (rows of 256 or 512
// columns with at most 4 heads: two tokens per warp).
template <typename T>
cudaError_t dispatch_fwd(const RouteArgs &a, cudaStream_t s)
{
    if (a.r != a.d) return cudaErrorNotSupported;
    const bool pair = a.H <= 4;  // two tokens per warp on rows of 256 or 512
    switch (a.d / 256) {
    case 1: return pair ? launch_fwd_pair<T, 1>(a, s) : launch_fwd_inst<T, 1, false>(a, s);
    case 2: return pair ? launch_fwd_pair<T, 2>(a, s) : launch_fwd_inst<T, 2, false>(a, s);
    case 3: return launch_fwd_inst<T, 3, false>(a, s);
    case 4: return launch_fwd_inst<T, 4, false>(a, s);
    case 5: return launch_fwd_inst<T, 5, false>(a, s);
    case 6: return launch_fwd_inst<T, 6, false>(a, s);
    case 7: return launch_fwd_inst<T, 7, false>(a, s);
    case 8: return launch_fwd_inst<T, 8, false>(a, s);
    default: return cudaErrorNotSupported;
    }
}

// Sliced keys, single pass, d = 256 * CPL with CPL in 1..10 (the
// sliced-key family's shapes; wider rows use its two-sweep forward).
template <typename T>
cudaError_t dispatch_fwd_sk(const RouteArgs &a, cudaStream_t s)
{
    switch (a.d / 256) {
    case 1: return launch_fwd_inst<T, 1, true>(a, s);
    case 2: return launch_fwd_inst<T, 2, true>(a, s);
    case 3: return launch_fwd_inst<T, 3, true>(a, s);
    case 4: return launch_fwd_inst<T, 4, true>(a, s);
    case 5: return launch_fwd_inst<T, 5, true>(a, s);
    case 6: return launch_fwd_inst<T, 6, true>(a, s);
    case 7: return launch_fwd_inst<T, 7, true>(a, s);
    case 8: return launch_fwd_inst<T, 8, true>(a, s);
    case 9: return launch_fwd_inst<T, 9, true>(a, s);
    case 10: return launch_fwd_inst<T, 10, true>(a, s);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace ar

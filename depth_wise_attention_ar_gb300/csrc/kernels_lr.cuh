// Routing kernels for sliced keys (r < d): "Low-Rank Attention Residuals",
// Sec. 3.2-3.3 (Eq. 8-12, keys = RMSNorm of the last r coordinates, values
// full width), with MHAR heads laid over the key slice (head h scores with
// the h-th r/H block of the key and mixes the h-th d/H block of the value).
//
// Forward, per warp and token (two sweeps, exact softmax), for rows wider
// than 2560 (narrower rows take the single-pass sliced-key forward of
// kernels_fwd.cuh):
//   sweep 1: the key tails of the N listed rows (r coordinates each) land in a
//            per-warp shared-memory cache by 1-D bulk copies; every head's
//            scores, softmax weights and lse follow from the cache;
//   sweep 2: the value rows are mixed in column blocks of CW columns (at most
//            1024; CW divides both d - r and r) with those weights: blocks left
//            of the tail stream through a ring of shared-memory stages, tail
//            blocks come from the cache, so every source coordinate is read
//            from HBM once.
//   The cache is double-buffered: the next token's key tails are requested as
//   soon as this token's weights are known, and arrive during sweep 2.
// Backward, per warp, over an even contiguous share of the (token, source)
// items (token-major): G = dL/dout of the current token sits in registers
// when the chunk count d/256 is a template constant (rows up to 2560 wide),
// else in shared memory; a stage holds the source row and (unless first
// touch) its fp32 gradient row. Pass A: value dot P (head's value slice) and
// raw score zr (head's key slice). Pass B: the key-path terms are added into
// the staged gradient row on the tail. Pass C: w*G is added on every
// coordinate (and the radial term outside the slice for the full-width
// norm) and the row is written out. On bf16 rows up to 2048 wide with key
// tails up to half the row, the next token's G, output chunks, lse and first
// inverse RMS values are loaded into registers while this token's items run.
#pragma once

#include "common.cuh"
#include "launch_util.cuh"
#include "shapes.h"

namespace ar {

template <typename T, int KMAX>
__global__ void __launch_bounds__(32) route_fwd_lr_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    constexpr int S = kLrFwdStages;
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x;
    const int d = a.d, r = a.r, N = a.n_src, H = a.H;
    const int64_t TT = a.T;
    const int CW = lr_block_cols(d, r);             // columns per block
    const int cwc = CW / 8;                         // chunks per block
    const uint32_t eb = (uint32_t)sizeof(T);
    const uint32_t key_bytes = (uint32_t)r * eb, blk_bytes = (uint32_t)CW * eb;
    const int nblk_v = (d - r) / CW, nblk_k = r / CW;  // value-only and tail blocks

    for (int i = lane; i < N; i += 32) s_rows[i] = a.rows[i];
    unsigned char *kc = smem;                                        // [2][N][r]
    unsigned char *ring = kc + 2 * (size_t)N * key_bytes;            // [S][CW]
    float *zs = reinterpret_cast<float *>(ring + (size_t)S * blk_bytes);  // [N][H]
    float *ws = zs + (size_t)N * H;                                  // [N][H]
    uint64_t *kbar = reinterpret_cast<uint64_t *>(ws + (size_t)N * H);
    uint64_t *rbar = kbar + 2;
    float *inv2 = reinterpret_cast<float *>(rbar + S);               // [2][256]
    if (lane == 0) {
        mbar_init(&kbar[0], 1);
        mbar_init(&kbar[1], 1);
        for (int s = 0; s < S; ++s) mbar_init(&rbar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int LPH = 32 / H;
    const int h = lane / LPH, sub = lane - h * LPH;
    const int K = d / H;                            // value slice width
    // key chunks of this lane (relative to the first key coordinate): chunk
    // sub + LPH*j of its head's r/(8H) key chunks, where that exists
    const int ckh = r / 8 / H;
    int kidx[KMAX];
    bool kval[KMAX];
    float qg[KMAX][8];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        kval[j] = sub + LPH * j < ckh;
        kidx[j] = h * ckh + sub + LPH * j;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = kidx[j] * 8 + e;
            qg[j][e] = kval[j] ? ldg_chk(a.q + c * a.q_stride) * (a.g ? ldg_chk(a.g + c * a.g_stride) : 1.0f) : 0.f;
        }
    }

    const int64_t GW = gridDim.x, gw = blockIdx.x;
    const int64_t ntok = gw < TT ? (TT - 1 - gw) / GW + 1 : 0;
    const uint64_t pol = l2_policy_evict_first();
    const unsigned char *bank = static_cast<const unsigned char *>(a.bank);
    const uint64_t row_bytes = (uint64_t)d * eb;

    auto issue_keys = [&](int64_t k) {  // key tails of token k -> cache k % 2
        if (lane == 0) {
            const int64_t tok = gw + k * GW;
            unsigned char *dst = kc + (size_t)(k & 1) * N * key_bytes;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&kbar[k & 1], key_bytes * (uint32_t)N);
            for (int n = 0; n < N; ++n)
                bulk_g2s(dst + (size_t)n * key_bytes,
                         bank + ((int64_t)s_rows[n] * TT + tok) * row_bytes + (uint64_t)(d - r) * eb,
                         key_bytes, &kbar[k & 1], pol);
        }
    };
    // value ring: items (token k, value block b, source n), n fastest
    const int64_t per_tok = (int64_t)nblk_v * N;
    const int64_t total = ntok * per_tok;
    int64_t issued = 0, k_p = 0;
    int b_p = 0, n_p = 0, slot_p = 0;
    auto issue_next = [&]() {
        if (lane == 0) {
            const int64_t tok = gw + k_p * GW;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&rbar[slot_p], blk_bytes);
            bulk_g2s(ring + (size_t)slot_p * blk_bytes,
                     bank + ((int64_t)s_rows[n_p] * TT + tok) * row_bytes + (uint64_t)b_p * blk_bytes,
                     blk_bytes, &rbar[slot_p], pol);
        }
        ++issued;
        if (++n_p == N) {
            n_p = 0;
            if (++b_p == nblk_v) { b_p = 0; ++k_p; }
        }
        if (++slot_p == S) slot_p = 0;
    };
    auto load_inv = [&](int64_t k, float *dst) {
        const int64_t tok = gw + k * GW;
        for (int nn = lane; nn < N; nn += 32) dst[nn] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[nn]);
    };

    if (ntok > 0) {
        issue_keys(0);
        load_inv(0, inv2);
    }
    for (int s = 0; s < S && issued < total; ++s) issue_next();

    uint32_t kphase = 0, rphase = 0;
    int slot = 0;
    bool ok = true;
    int64_t consumed = 0;
    for (int64_t k = 0; k < ntok && ok; ++k) {
        const int64_t tok = gw + k * GW;
        const int buf = (int)(k & 1);
        float *cinv = inv2 + buf * AR_MAX_SOURCES;
        __syncwarp();
        // ---- sweep 1: scores of every (source, head) from the key cache
        const bool got = mbar_wait(&kbar[buf], (kphase >> buf) & 1u, kWaitLimit);
        if (!__all_sync(FULL, got)) { ok = false; break; }
        kphase ^= 1u << buf;
        const unsigned char *keys = kc + (size_t)buf * N * key_bytes;
        for (int n = 0; n < N; ++n) {
            const T *kr = reinterpret_cast<const T *>(keys + (size_t)n * key_bytes);
            float zr = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (kval[j]) {
                    float v[8];
                    ld_chunk_s(kr + kidx[j] * 8, v);
                    zr = __fadd_rn(zr, dot8(qg[j], v));
                }
            }
            zr = group_sum(zr, LPH);
            if (sub == 0) zs[n * H + h] = __fmul_rn(zr, cinv[n]);
        }
        __syncwarp();
        if (sub == 0) {  // exact softmax over the N sources of head h
            float m = zs[h];
            for (int n = 1; n < N; ++n) m = fmaxf(m, zs[n * H + h]);
            float l = 0.f;
            for (int n = 0; n < N; ++n) l += exp2f((zs[n * H + h] - m) * kLog2e);
            const float rl = 1.f / l;
            for (int n = 0; n < N; ++n) ws[n * H + h] = exp2f((zs[n * H + h] - m) * kLog2e) * rl;
            st_chk(a.lse + (tok * H + h), m + log2f(l) * kLn2);
        }
        __syncwarp();
        // the next token's keys and inverse RMS can come in now
        if (k + 1 < ntok) {
            issue_keys(k + 1);
            load_inv(k + 1, inv2 + (1 - buf) * AR_MAX_SOURCES);
        }
        // ---- sweep 2: mix column blocks with the weights
        for (int b = 0; b < nblk_v + nblk_k && ok; ++b) {
            float acc[4][8];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
            const bool tail = b >= nblk_v;
            for (int n = 0; n < N; ++n) {
                const unsigned char *src;
                if (tail) {
                    src = keys + (size_t)n * key_bytes + (size_t)(b - nblk_v) * blk_bytes;
                } else {
                    const bool g2 = mbar_wait(&rbar[slot], (rphase >> slot) & 1u, kWaitLimit);
                    if (!__all_sync(FULL, g2)) { ok = false; break; }
                    rphase ^= 1u << slot;
                    src = ring + (size_t)slot * blk_bytes;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = lane + 32 * j;                   // chunk within the block
                    if (c < cwc) {
                        const int col = b * CW + c * 8;
                        const float wn = ws[n * H + col / K];
                        float v[8];
                        ld_chunk_s(reinterpret_cast<const T *>(src) + c * 8, v);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(wn, v[e], acc[j][e]);
                    }
                }
                if (!tail) {
                    __syncwarp();
                    ++consumed;
                    if (issued < total) issue_next();
                    if (++slot == S) slot = 0;
                }
            }
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (lane + 32 * j < cwc)
                    store_output<T>(a, tok * d + b * CW + (lane + 32 * j) * 8, acc[j]);
        }
    }
    if (!ok) {
        if (lane == 0) report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
        for (int64_t j = consumed; j < issued; ++j) {
            mbar_wait(&rbar[slot], (rphase >> slot) & 1u, kDrainLimit);
            rphase ^= 1u << slot;
            if (++slot == S) slot = 0;
        }
        mbar_wait(&kbar[0], kphase & 1u, kDrainLimit);
        mbar_wait(&kbar[1], (kphase >> 1) & 1u, kDrainLimit);
    }
}

inline size_t lr_bwd_smem_bytes(int d, size_t esize, bool g_in_registers)
{
    return (size_t)kLrBwdStages * ((size_t)d * esize + (size_t)d * 4)  // ring
           + (g_in_registers ? 0 : (size_t)d * esize)                   // G of the token
           + (size_t)kLrBwdStages * 8 + (size_t)AR_MAX_SOURCES * 4;
}

template <typename T, int KMAX, int CPLT = 0>
__global__ void __launch_bounds__(32) route_bwd_lr_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    __shared__ uint32_t s_first[AR_MAX_SOURCES / 32];
    constexpr int S = kLrBwdStages;
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x;
    const int d = a.d, r = a.r, N = a.n_src, H = a.H;
    const int64_t TT = a.T;
    const uint32_t vbytes = (uint32_t)d * (uint32_t)sizeof(T), gbytes = (uint32_t)d * 4u;
    const uint32_t slot_bytes = vbytes + gbytes;

    for (int i = lane; i < N; i += 32) s_rows[i] = a.rows[i];
    if (lane < AR_MAX_SOURCES / 32) s_first[lane] = a.first_mask[lane];
    unsigned char *ring = smem;
    T *Gs = reinterpret_cast<T *>(ring + (size_t)S * slot_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<unsigned char *>(Gs) +
                                                  (CPLT > 0 ? 0u : vbytes));
    float *cur_inv = reinterpret_cast<float *>(bars + S);
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int LPH = 32 / H;
    const int h = lane / LPH, sub = lane - h * LPH;
    const int cpl = CPLT > 0 ? CPLT : d / 256;      // value chunks per lane
    const int key0 = (d - r) / 8;                   // first key chunk
    // With the chunk count a template constant (CPLT > 0) the chunk loops
    // unroll and the token's G stays in registers (Gr) instead of shared
    // memory; the arithmetic and its order are the same either way.
    float Gr[CPLT > 0 ? CPLT : 1][8];
    auto for_chunks = [&](auto &&f) {
        if constexpr (CPLT > 0) {
#pragma unroll
            for (int j = 0; j < CPLT; ++j) f(j);
        } else {
            for (int j = 0; j < cpl; ++j) f(j);
        }
    };
    const int ckh = r / 8 / H;                      // key chunks per head
    int kidx[KMAX];
    bool kval[KMAX];
    float qg[KMAX][8], U[KMAX][8];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        kval[j] = sub + LPH * j < ckh;
        kidx[j] = key0 + h * ckh + sub + LPH * j;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = (kidx[j] - key0) * 8 + e;
            qg[j][e] = kval[j] ? ldg_chk(a.q + c * a.q_stride) * (a.g ? ldg_chk(a.g + c * a.g_stride) : 1.0f) : 0.f;
            U[j][e] = 0.f;
        }
    }
    // value chunk j of this lane: h * (cpl * LPH) + sub + LPH * j
    const int vbase = h * cpl * LPH + sub;
    const float inv_width = 1.0f / (float)(a.norm_full ? d : r);

    const int64_t GW = gridDim.x, gw = blockIdx.x;
    const int64_t total = TT * N;
    const int64_t lo = total * gw / GW, hi = total * (gw + 1) / GW;
    const uint64_t pol = l2_policy_evict_first();

    int64_t issued = lo, tok_p = lo / N;
    int n_p = (int)(lo - tok_p * N), slot_p = 0;
    auto issue_next = [&]() {
        if (lane == 0) {
            const bool first = (s_first[n_p >> 5] >> (n_p & 31)) & 1u;
            const int64_t off = (int64_t)s_rows[n_p] * TT + tok_p;
            unsigned char *dst = ring + (size_t)slot_p * slot_bytes;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[slot_p], vbytes + (first ? 0u : gbytes));
            bulk_g2s(dst, static_cast<const unsigned char *>(a.bank) + off * vbytes, vbytes,
                     &bars[slot_p], pol);
            if (!first) bulk_g2s(dst + vbytes, a.grad + off * d, gbytes, &bars[slot_p], pol);
        }
        ++issued;
        if (++n_p == N) { n_p = 0; ++tok_p; }
        if (++slot_p == S) slot_p = 0;
    };
    for (int s = 0; s < S && issued < hi; ++s) issue_next();

    // delta form: G = alpha dL/dh enters linearly, so G stays in the storage
    // dtype and alpha scales the dot products and the w G term
    float S_h = 0.f, lse_h = 0.f, dal = 0.f;
    const float alpha = a.alpha ? ldg_chk(a.alpha) : 1.0f;
    int64_t tok = lo / N, i = lo;
    int n = (int)(lo - tok * N), slot = 0;
    uint32_t phase = 0;
    bool ok = true;

    // bf16 rows of up to 2048 columns with a constant chunk count: the next
    // token's G and forward output chunks, lse and (first 32 sources) inverse
    // RMS are loaded into registers while this token's items run, so a token
    // start does not wait on DRAM. (GB300, 49 sites, T = 4096: backward
    // 3.24 -> 3.18 ms at d = 1536; at d = 2560 the longer items hide the wait
    // already and the extra registers cost 9.41 -> 9.53 ms, so not there;
    // nor with key tails over half the row, where the registers would spill.)
    constexpr bool kPre = CPLT > 0 && CPLT <= 8 && 2 * KMAX <= CPLT + 1 && sizeof(T) == 2;
    uint4 preG[kPre ? CPLT : 1], preO[kPre ? CPLT : 1];
    float pre_lse = 0.f, pre_inv = 0.f;
    const int64_t last_tok = hi > lo ? (hi - 1) / N : -1;
    auto prefetch_tok = [&](int64_t t) {
        if constexpr (kPre) {
            const uint4 *g4 = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.dout) + t * d);
            const uint4 *o4 = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.fout) + t * d);
#pragma unroll
            for (int j = 0; j < CPLT; ++j) {
                const int c = vbase + LPH * j;
                preG[j] = ldg16_chk(g4 + c);
                preO[j] = ldg16_chk(o4 + c);
            }
            pre_lse = ldg_chk(a.lse + t * H + h);
            if (lane < N) pre_inv = ldg_chk(a.inv + t * a.inv_ld + s_rows[lane]);
        }
    };
    if (tok <= last_tok) prefetch_tok(tok);

    for (; i < hi; ++i) {
        if (i == lo || n == 0) {
            __syncwarp();
            const T *grow = static_cast<const T *>(a.dout) + tok * d;
            const T *orow = static_cast<const T *>(a.fout) + tok * d;
            float sp = 0.f;
            for_chunks([&](int j) {
                const int c = vbase + LPH * j;
                float gv[8], o[8];
                if constexpr (kPre) {
                    unpack_bf16x8(preG[j], gv);
                    unpack_bf16x8(preO[j], o);
                } else {
                    const uint4 graw = ldg16_chk(reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const unsigned char *>(grow) + (size_t)c * ChunkBytes<T>::value));
                    if constexpr (sizeof(T) == 2) {
                        if constexpr (CPLT == 0) *reinterpret_cast<uint4 *>(Gs + c * 8) = graw;
                        unpack_bf16x8(graw, gv);
                    } else {
                        const uint4 g2 = ldg16_chk(reinterpret_cast<const uint4 *>(
                            reinterpret_cast<const unsigned char *>(grow) + (size_t)c * 32 + 16));
                        if constexpr (CPLT == 0) {
                            reinterpret_cast<uint4 *>(Gs + c * 8)[0] = graw;
                            reinterpret_cast<uint4 *>(Gs + c * 8)[1] = g2;
                        }
                        gv[0] = __uint_as_float(graw.x); gv[1] = __uint_as_float(graw.y);
                        gv[2] = __uint_as_float(graw.z); gv[3] = __uint_as_float(graw.w);
                        gv[4] = __uint_as_float(g2.x); gv[5] = __uint_as_float(g2.y);
                        gv[6] = __uint_as_float(g2.z); gv[7] = __uint_as_float(g2.w);
                    }
                    ld_chunk_g(orow + c * 8, o);
                }
                if constexpr (CPLT > 0) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) Gr[j][e] = gv[e];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) sp = fmaf(gv[e], o[e], sp);
            });
            // each token's <dL/dh, routed> counted by the warp owning (t, 0)
            if (a.dalpha && n == 0) dal += warp_sum(sp);
            S_h = a.coupling ? ldg_chk(a.coupling + (tok * H + h)) : alpha * group_sum(sp, LPH);
            if constexpr (kPre) {
                lse_h = pre_lse;
                if (lane < N) cur_inv[lane] = pre_inv;
                for (int nn = lane + 32; nn < N; nn += 32)
                    cur_inv[nn] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[nn]);
                if (tok < last_tok) prefetch_tok(tok + 1);
            } else {
                lse_h = ldg_chk(a.lse + tok * H + h);
                for (int nn = lane; nn < N; nn += 32)
                    cur_inv[nn] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[nn]);
            }
            __syncwarp();
        }
        const bool got = mbar_wait(&bars[slot], (phase >> slot) & 1u, kWaitLimit);
        if (!__all_sync(FULL, got)) { ok = false; break; }
        phase ^= 1u << slot;
        unsigned char *vb = ring + (size_t)slot * slot_bytes;
        const T *V = reinterpret_cast<const T *>(vb);
        float *gb = reinterpret_cast<float *>(vb + vbytes);
        const bool first = (s_first[n >> 5] >> (n & 31)) & 1u;

        // pass A: value dot and raw score
        float P = 0.f, zr = 0.f;
        for_chunks([&](int j) {
            const int c = vbase + LPH * j;
            float v[8];
            ld_chunk_s(V + c * 8, v);
            if constexpr (CPLT > 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) P = fmaf(Gr[j][e], v[e], P);
            } else {
                float gv[8];
                ld_chunk_s(Gs + c * 8, gv);
#pragma unroll
                for (int e = 0; e < 8; ++e) P = fmaf(gv[e], v[e], P);
            }
        });
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (kval[j]) {
                float v[8];
                ld_chunk_s(V + kidx[j] * 8, v);
                zr = __fadd_rn(zr, dot8(qg[j], v));
            }
        }
        P = alpha * group_sum(P, LPH);
        zr = group_sum(zr, LPH);
        const float iv = cur_inv[n];
        const float w = exp2f((__fmul_rn(iv, zr) - lse_h) * kLog2e);
        const float dz = w * (P - S_h);
        const float C = (H == 1) ? dz * zr : warp_sum(sub == 0 ? dz * zr : 0.f);
        const float coef = iv * iv * iv * C * inv_width;
        const float ak = iv * dz;
        const float wa = w * alpha;

        // pass B: key-path terms on the tail, into the staged gradient row
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (!kval[j]) continue;
            float v[8], nv[8];
            ld_chunk_s(V + kidx[j] * 8, v);
            if (first) {
#pragma unroll
                for (int e = 0; e < 8; ++e) nv[e] = 0.f;
            } else {
                ld_chunk_s(gb + kidx[j] * 8, nv);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                nv[e] = fmaf(ak, qg[j][e], nv[e]);
                nv[e] = fmaf(-coef, v[e], nv[e]);
                U[j][e] = fmaf(ak, v[e], U[j][e]);
            }
            st_f32x8_s(gb + kidx[j] * 8, nv);
        }
        __syncwarp();
        // pass C: w G everywhere (+ radial term off the slice for the full norm)
        float *grad_row = a.grad + ((int64_t)s_rows[n] * TT + tok) * d;
        const float cv = a.norm_full ? coef : 0.f;
        for_chunks([&](int j) {
            const int c = vbase + LPH * j;
            const bool tail = c >= key0;
            float nv[8], gv[8];
            if (tail || !first) {
                ld_chunk_s(gb + c * 8, nv);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) nv[e] = 0.f;
            }
            if constexpr (CPLT > 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) gv[e] = Gr[j][e];
            } else {
                ld_chunk_s(Gs + c * 8, gv);
            }
            if (!tail && cv != 0.f) {
                float v[8];
                ld_chunk_s(V + c * 8, v);
#pragma unroll
                for (int e = 0; e < 8; ++e) nv[e] = fmaf(-cv, v[e], nv[e]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) nv[e] = fmaf(wa, gv[e], nv[e]);
            st_grad8(grad_row + c * 8, 0, nv, a.grad_v8);
        });
        __syncwarp();
        if (issued < hi) issue_next();
        if (++n == N) { n = 0; ++tok; }
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
    float *wrow = a.ws + gw * r;
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
        if (kval[j]) st_f32x8_g(wrow + (kidx[j] - key0) * 8, U[j]);
    if (a.dalpha && lane == 0) {
        AR_GUARD_G(a.ws + GW * r + gw * 4, 16, true, 16, return)
        *reinterpret_cast<float4 *>(a.ws + GW * r + gw * 4) = make_float4(dal, 0.f, 0.f, 0.f);
    }
}

template <typename T, int KMAX>
cudaError_t launch_lr_fwd_inst(const RouteArgs &a, cudaStream_t s)
{
    const void *k = reinterpret_cast<const void *>(&route_fwd_lr_kernel<T, KMAX>);
    const size_t smem = lr_fwd_smem_bytes(a.d, a.r, a.n_src, a.H, sizeof(T));
    if (smem > 200 * 1024) return cudaErrorNotSupported;
    int grid = 0;
    cudaError_t e = persistent_grid(k, 32, smem, &grid);
    if (e != cudaSuccess) return e;
    route_fwd_lr_kernel<T, KMAX><<<grid, 32, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int KMAX, int CPLT = 0>
cudaError_t lr_bwd_inst(const RouteArgs *a, cudaStream_t s, int *grid_warps)
{
    const void *k = reinterpret_cast<const void *>(&route_bwd_lr_kernel<T, KMAX, CPLT>);
    const size_t smem = lr_bwd_smem_bytes(a->d, sizeof(T), CPLT > 0);
    int grid = 0;
    cudaError_t e = persistent_grid(k, 32, smem, &grid);
    if (e != cudaSuccess) return e;
    if (grid_warps) {
        *grid_warps = grid;
        return cudaSuccess;
    }
    route_bwd_lr_kernel<T, KMAX, CPLT><<<grid, 32, smem, s>>>(*a);
    return cudaGetLastError();
}

// Key chunks per lane (at most): ceil(r / 256). Served: r a multiple of 8 with
// r/H a multiple of 8, r <= d <= 4096 with d a multiple of 256.

#define AR_LR_KMAX_CASES(X) X(1) X(2) X(3) X(4) X(5) X(6) X(8) X(10) X(12) X(14) X(16)

template <typename T>
cudaError_t dispatch_lr_fwd(const RouteArgs &a, cudaStream_t s)
{
    const int km = lr_kmax(a.r);
#define AR_CASE(K) if (km <= K) return launch_lr_fwd_inst<T, K>(a, s);
    AR_LR_KMAX_CASES(AR_CASE)
#undef AR_CASE
    return cudaErrorNotSupported;
}

// Rows up to 2560 wide: the chunk count d / 256 as a template constant, with
// the key chunks per lane held in the smallest of a quarter, a half or all of
// it that fits ceil(r / 256). Instantiated in its own translation units.
template <typename T, int CPL>
cudaError_t lr_bwd_fixed(const RouteArgs *a, cudaStream_t s, int *grid_warps)
{
    constexpr int kQuarter = (CPL + 3) / 4, kHalf = (CPL + 1) / 2;
    const int km = lr_kmax(a->r);
    if (km <= kQuarter) return lr_bwd_inst<T, kQuarter, CPL>(a, s, grid_warps);
    if (km <= kHalf) return lr_bwd_inst<T, kHalf, CPL>(a, s, grid_warps);
    // key tails over half of rows 2304 or 2560 wide: G and the key chunks
    // together would spill, so the chunk loop stays a runtime loop there
    if constexpr (CPL >= 9)
        return lr_bwd_inst<T, 10, 0>(a, s, grid_warps);
    else
        return lr_bwd_inst<T, CPL, CPL>(a, s, grid_warps);
}

template <typename T>
cudaError_t dispatch_lr_bwd_fixed(const RouteArgs *a, cudaStream_t s, int *grid_warps)
{
    switch (a->d / 256) {
    case 1: return lr_bwd_fixed<T, 1>(a, s, grid_warps);
    case 2: return lr_bwd_fixed<T, 2>(a, s, grid_warps);
    case 3: return lr_bwd_fixed<T, 3>(a, s, grid_warps);
    case 4: return lr_bwd_fixed<T, 4>(a, s, grid_warps);
    case 5: return lr_bwd_fixed<T, 5>(a, s, grid_warps);
    case 6: return lr_bwd_fixed<T, 6>(a, s, grid_warps);
    case 7: return lr_bwd_fixed<T, 7>(a, s, grid_warps);
    case 8: return lr_bwd_fixed<T, 8>(a, s, grid_warps);
    case 9: return lr_bwd_fixed<T, 9>(a, s, grid_warps);
    case 10: return lr_bwd_fixed<T, 10>(a, s, grid_warps);
    default: return cudaErrorNotSupported;
    }
}

template <typename T>
cudaError_t dispatch_lr_bwd(const RouteArgs *a, cudaStream_t s, int *grid_warps)
{
    if (a->d / 256 <= 10) return dispatch_lr_bwd_fixed<T>(a, s, grid_warps);
    const int km = lr_kmax(a->r);
#define AR_CASE(K) if (km <= K) return lr_bwd_inst<T, K>(a, s, grid_warps);
    AR_LR_KMAX_CASES(AR_CASE)
#undef AR_CASE
    return cudaErrorNotSupported;
}

}  // namespace ar

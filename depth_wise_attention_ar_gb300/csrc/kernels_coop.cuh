// Routing kernels for wide rows: four warps of a block share every item.
//
// Same mathematics as the full-key kernels ("Multi-Head Attention Residuals",
// Eq. 3 and Appendix E; "Low-Rank Attention Residuals", Eq. 8-13 and 15-22),
// for rows too wide for one warp's registers (d > 2048) and for sliced keys
// on wide rows. The row is split into four column groups of CG = d/4 columns;
// warp w owns group w and whole value heads (H/4 of them). One staged row
// (source row, plus its fp32 gradient row in the backward) is shared by the
// block; thread 0 refills a stage once all four warps are past it.
//
// Key handling
// - r = d (full keys): a warp's key heads are its value heads, so the
//   forward needs no exchange; the backward sums the RMS coupling term
//   sum_h dz*zr over the four warps through shared memory.
// - r < d (sliced keys, r a multiple of CG): the key tail lies in the last
//   r/CG warps' column groups. In the forward those warps compute every
//   head's raw score and publish it. In the backward every warp scores its own
//   heads from their key slices and stages their key-path terms in the shared
//   gradient row; the warps owning the tail wait for them on a named barrier
//   before they write it. The forward's and the backward's scores then differ
//   in summation order (they agree to rounding); with full keys both take the
//   same lanes and order, so the bits match.
//
// The forward takes one block barrier per item and can take the site's append
// (FRESH): the new row's item stages the row it is formed from, each warp
// forms its columns (a copy, or a block partial sum rounded once) into the
// stage and the row's slot, and the item's barrier publishes the squares for
// the new row's inverse RMS. In the delta form, and for a fused partial sum,
// a per-token row (the residual stream, or the sublayer output to add) is
// staged by a bulk copy at the token's first item.
#pragma once

#include "common.cuh"
#include "launch_util.cuh"

namespace ar {

constexpr int kCoopWarps = 4;
constexpr int kCoopFwdStages = 4;
// Backward stages of (row + fp32 gradient row), and with bf16 rows a block
// buffer (2 d b bytes) into which each thread fetches its own chunks of the
// next token's dL/dout and output rows by cp.async while the current token
// runs. bf16 rows take 2 stages and the buffer, which leaves room for three
// blocks of d = 4096 (full keys 161 registers, sliced keys 160). Against 3
// stages with an L2 prefetch of the next token's rows: delta 8B backward
// 20.47 -> 19.54 ms; low-rank block 19.00 -> 18.44 ms together with the
// balanced key work below (4 stages and the buffer left one block per SM:
// 28.9 ms).
constexpr int coop_bwd_stages(size_t esize, bool lr) { return esize == 2 ? 2 : 3; }
constexpr bool coop_bwd_tokbuf(size_t esize) { return esize == 2; }

struct CoopMap {
    int Hw, LPH, hl, sub, h;      // value heads per warp, lanes per head, local head, lane in head, head
    int kw, Hk, LPHk, hk, ksub;   // key warps, key heads per key warp, lanes per key head, key head
    bool key_warp;
};

__device__ __forceinline__ CoopMap coop_map(int w, int lane, int H, int d, int r)
{
    CoopMap m;
    m.Hw = H / kCoopWarps;
    m.LPH = 32 / m.Hw;
    m.hl = lane / m.LPH;
    m.sub = lane - m.hl * m.LPH;
    m.h = w * m.Hw + m.hl;
    const int CG = d / kCoopWarps;
    m.kw = r / CG;
    m.Hk = H / m.kw;
    m.LPHk = 32 / m.Hk;
    const int kwi = w - (kCoopWarps - m.kw);
    m.key_warp = kwi >= 0;
    m.hk = m.key_warp ? kwi * m.Hk + lane / m.LPHk : 0;
    m.ksub = lane % m.LPHk;
    return m;
}

// Stages, barriers, scores, inverse RMS; with the delta form also two
// buffers of the residual-stream row and their barriers.
// Stages, barriers, scores, inverse RMS, the fused append's squares; with
// the delta form or a fused partial sum also two buffers of a per-token row
// (the residual stream, or the sublayer output to add) and their barriers.
inline size_t coop_fwd_smem_bytes(int d, size_t esize, bool tok_row)
{
    return (size_t)kCoopFwdStages * d * esize + kCoopFwdStages * 8 + 2 * 32 * 4 +
           2 * AR_MAX_SOURCES * 4 + 8 * 4 + (tok_row ? 16 + 2 * (size_t)d * esize : 0);
}

template <typename T, int CPL, bool LR, bool FRESH = false>
__global__ void __launch_bounds__(kCoopWarps * 32)
    route_fwd_coop_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    constexpr int S = kCoopFwdStages;
    constexpr int CB = ChunkBytes<T>::value;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, r = a.r, N = a.n_src, H = a.H;
    const int64_t TT = a.T;
    const uint32_t row_bytes = (uint32_t)d * (uint32_t)sizeof(T);

    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    unsigned char *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)S * row_bytes);
    float *zs = reinterpret_cast<float *>(bars + S);   // [2][32] scores per head
    float *cur_inv = zs + 64;                           // [2][AR_MAX_SOURCES]
    float *ssq = cur_inv + 2 * AR_MAX_SOURCES;           // [2][4] fused append: squares
    // a per-token row staged by a bulk copy at the token's first item (two
    // buffers, by token parity): the delta form's residual stream, or the
    // sublayer output a fused partial sum adds
    const bool delta = a.partial != nullptr;
    const bool fresh_acc = FRESH && a.acc_row >= 0;
    const bool tok_row = delta || fresh_acc;
    const unsigned char *tok_src = static_cast<const unsigned char *>(delta ? a.partial : a.fresh_src);
    uint64_t *pbars = reinterpret_cast<uint64_t *>(ssq + 8);
    unsigned char *pbuf = reinterpret_cast<unsigned char *>(pbars + 2);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        if (tok_row) {
            mbar_init(&pbars[0], 1);
            mbar_init(&pbars[1], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    const CoopMap mp = coop_map(w, lane, H, d, r);
    const int gchunk = w * CPL * 32;                    // first chunk of this warp's group
    int cidx[CPL], kidx[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        cidx[j] = gchunk + chunk_of<CPL>(mp.hl, mp.sub, mp.LPH, j);
        kidx[j] = gchunk + chunk_of<CPL>(mp.hk % mp.Hk, mp.ksub, mp.LPHk, j);
    }
    const int key0 = (d - r) / 8;
    float qg[CPL][8];
#pragma unroll
    for (int j = 0; j < CPL; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = (LR ? kidx[j] : cidx[j]) * 8 + e - key0 * 8;
            const bool have = !LR || mp.key_warp;
            qg[j][e] = have ? ldg_chk(a.q + c * a.q_stride) * (a.g ? ldg_chk(a.g + c * a.g_stride) : 1.0f) : 0.f;
        }

    const int64_t GB = gridDim.x, gb = blockIdx.x;
    const int64_t ntok = gb < TT ? (TT - 1 - gb) / GB + 1 : 0;
    const int64_t total = ntok * N;
    const uint64_t pol = l2_policy_evict_first();

    int64_t issued = 0, tok_p = gb;
    int n_p = 0, slot_p = 0;
    auto issue_next = [&]() {
        if (threadIdx.x == 0) {
            // the fused append's item stages the row the new one is formed
            // from: the previous partial sum, or the source to copy
            const unsigned char *src = static_cast<const unsigned char *>(a.bank) +
                                       ((int64_t)s_rows[n_p] * TT + tok_p) * row_bytes;
            if (FRESH && n_p + 1 == a.fresh1 && a.fresh_src)
                src = a.acc_row >= 0
                          ? static_cast<const unsigned char *>(a.bank) +
                                ((int64_t)a.acc_row * TT + tok_p) * row_bytes
                          : static_cast<const unsigned char *>(a.fresh_src) + tok_p * row_bytes;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[slot_p], row_bytes);
            bulk_g2s(ring + (size_t)slot_p * row_bytes, src, row_bytes, &bars[slot_p], pol);
        }
        ++issued;
        if (++n_p == N) { n_p = 0; tok_p += GB; }
        if (++slot_p == S) slot_p = 0;
    };
    for (int s = 0; s < S && issued < total; ++s) issue_next();

    // One block barrier per item: it carries the stage wait's outcome, the
    // key warp's scores (sliced keys) and the token's inverse RMS, and shows
    // that every warp is past the previous item, whose stage thread 0 then
    // refills. Scores and inverse RMS are double-buffered for that.
    int n = 0, slot = 0, par = 0, tpar = 0;
    uint32_t phase = 0, pphase = 0;
    int64_t tok = gb, i = 0;
    float m = 0.f, l = 0.f;
    float acc[CPL][8];
    const float alpha = delta && a.alpha ? ldg_chk(a.alpha) : 1.0f;
    bool ok = true, bad = false;
    for (; i < total; ++i) {
        float *inv_t = cur_inv + tpar * AR_MAX_SOURCES;
        if (n == 0) {
            // every warp is past token tok - 2 GB, whose row used this buffer
            if (tok_row && threadIdx.x == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&pbars[tpar], row_bytes);
                bulk_g2s(pbuf + (size_t)tpar * row_bytes, tok_src + tok * row_bytes, row_bytes,
                         &pbars[tpar], pol);
            }
            for (int nn = threadIdx.x; nn < N; nn += blockDim.x)
                inv_t[nn] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[nn]);
        }
        const bool got = mbar_wait(&bars[slot], (phase >> slot) & 1u, kWaitLimit);
        const unsigned char *buf = ring + (size_t)slot * row_bytes;
        float v[CPL][8];
        const bool fresh = FRESH && n + 1 == a.fresh1;
        if constexpr (FRESH) {
            if (fresh && got) {
                // the fused append: form the new row where needed (in the stage
                // and in its slot), then the squares of its stored values over
                // the RMS columns of this warp's group
                unsigned char *sb = ring + (size_t)slot * row_bytes;
                bool pg = true;
                if (fresh_acc) {
                    pg = mbar_wait(&pbars[tpar], (pphase >> tpar) & 1u, kWaitLimit);
                    pphase ^= 1u << tpar;
                    bad = bad || !pg;
                }
                if (a.fresh_src && pg) {
                    T *slot_row = static_cast<T *>(const_cast<void *>(a.bank)) +
                                  ((int64_t)s_rows[n] * TT + tok) * d;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) {
                        float x[8];
                        ld_chunk_s(reinterpret_cast<const T *>(sb + cidx[j] * CB), x);
                        if (fresh_acc) {
                            float y[8];
                            ld_chunk_s(reinterpret_cast<const T *>(pbuf + (size_t)tpar * row_bytes +
                                                                   cidx[j] * CB),
                                       y);
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[e] += y[e];
                        }
                        st_chunk_s(reinterpret_cast<T *>(sb + cidx[j] * CB), x);
                        st_chunk_g(slot_row + cidx[j] * 8, x);
                    }
                    __syncwarp();
                }
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    if (a.norm_full || cidx[j] >= key0) {
                        float x[8];
                        ld_chunk_s(reinterpret_cast<const T *>(sb + cidx[j] * CB), x);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
                    }
                }
                ss = warp_sum(ss);
                if (lane == 0) ssq[par * 4 + w] = ss;
            }
        }
        if constexpr (LR) {
            if (mp.key_warp && got) {
                float zr = 0.f;
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    float kv[8];
                    ld_chunk_s(reinterpret_cast<const T *>(buf + kidx[j] * CB), kv);
                    zr = __fadd_rn(zr, dot8(qg[j], kv));
                }
                zr = group_sum(zr, mp.LPHk);
                // the raw score: the inverse RMS is applied after the barrier
                if (mp.ksub == 0) zs[par * 32 + mp.hk] = zr;
            }
        }
        if (__syncthreads_or(!got || bad)) { ok = false; break; }
        phase ^= 1u << slot;
        if (i > 0 && issued < total) issue_next();  // the previous item's stage is free
        float iv = inv_t[n];
        if (FRESH && fresh) {
            const float sum = ((ssq[par * 4 + 0] + ssq[par * 4 + 1]) + ssq[par * 4 + 2]) + ssq[par * 4 + 3];
            iv = rsqrtf(fmaf(sum, 1.0f / (float)(a.norm_full ? d : r), a.eps));
            if (threadIdx.x == 0) st_chk(const_cast<float *>(a.inv) + (tok * a.inv_ld + s_rows[n]), iv);
        }

#pragma unroll
        for (int j = 0; j < CPL; ++j) ld_chunk_s(reinterpret_cast<const T *>(buf + cidx[j] * CB), v[j]);
        float z;
        if constexpr (!LR) {
            float zr = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) zr = __fadd_rn(zr, dot8(qg[j], v[j]));
            zr = group_sum(zr, mp.LPH);
            z = __fmul_rn(zr, iv);
        } else {
            z = __fmul_rn(zs[par * 32 + mp.h], iv);
        }
        if (n == 0) {
            m = z;
            l = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
        }
        const bool need = z > m + kRescaleTau;
        if (__any_sync(0xffffffffu, need)) {
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
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(p, v[j][e], acc[j][e]);

        if (n == N - 1) {
            const float rl = 1.f / l;
            bool pg = true;
            if (delta) {
                pg = mbar_wait(&pbars[tpar], (pphase >> tpar) & 1u, kWaitLimit);
                pphase ^= 1u << tpar;
                bad = bad || !pg;
            }
            if (pg) {
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = acc[j][e] * rl;
                    const int64_t off = tok * d + cidx[j] * 8;
                    if (delta) {
                        // out = partial + alpha * routed, routed kept for the backward
                        float pv[8], y[8];
                        ld_chunk_s(reinterpret_cast<const T *>(pbuf + (size_t)tpar * row_bytes +
                                                               cidx[j] * CB),
                                   pv);
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = fmaf(alpha, o[e], pv[e]);
                        if (a.routed) st_chunk_g(static_cast<T *>(a.routed) + off, o);
                        st_chunk_g(static_cast<T *>(a.out) + off, y);
                    } else {
                        store_output<T>(a, off, o);
                    }
                }
                if (mp.sub == 0) st_chk(a.lse + (tok * H + mp.h), m + log2f(l) * kLn2);
            }
        }
        par ^= 1;
        if (++n == N) {
            n = 0;
            tok += GB;
            tpar ^= 1;
        }
        if (++slot == S) slot = 0;
    }
    if (!ok || bad) {
        if (threadIdx.x == 0) {
            report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
            for (int64_t j = i; j < issued; ++j) {
                mbar_wait(&bars[slot], (phase >> slot) & 1u, kDrainLimit);
                phase ^= 1u << slot;
                if (++slot == S) slot = 0;
            }
            // a per-token row still in flight (the current token's)
            if (tok_row) mbar_wait(&pbars[tpar], (pphase >> tpar) & 1u, kDrainLimit);
        }
    }
}

inline size_t coop_bwd_smem_bytes(int d, size_t esize, bool lr)
{
    const size_t S = (size_t)coop_bwd_stages(esize, lr);
    const size_t base = S * ((size_t)d * esize + (size_t)d * 4) + S * 8 + 3 * 2 * 32 * 4;
    return coop_bwd_tokbuf(esize) ? (base + 15) / 16 * 16 + 2 * (size_t)d * esize : base;
}

template <typename T, int CPL, bool LR>
__global__ void __launch_bounds__(kCoopWarps * 32)
    route_bwd_coop_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    __shared__ uint32_t s_first[AR_MAX_SOURCES / 32];
    constexpr int S = coop_bwd_stages(sizeof(T), LR);
    constexpr int CB = ChunkBytes<T>::value;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, r = a.r, N = a.n_src, H = a.H;
    const int64_t TT = a.T;
    const uint32_t vbytes = (uint32_t)d * (uint32_t)sizeof(T), gbytes = (uint32_t)d * 4u;
    const uint32_t slot_bytes = vbytes + gbytes;

    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    for (int i = threadIdx.x; i < AR_MAX_SOURCES / 32; i += blockDim.x) s_first[i] = a.first_mask[i];
    unsigned char *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)S * slot_bytes);
    float *cws = reinterpret_cast<float *>(bars + S) + 128;  // [2][32] per-warp coupling sums
    constexpr bool kTok = coop_bwd_tokbuf(sizeof(T));
    T *tbuf = reinterpret_cast<T *>(smem + ((size_t)S * slot_bytes + S * 8 + 3 * 2 * 32 * 4 + 15) / 16 * 16);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const CoopMap mp = coop_map(w, lane, H, d, r);
    const int sw = ((lane >> 2) & 1) * 4;
    const int gchunk = w * CPL * 32;
    int cidx[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) cidx[j] = gchunk + chunk_of<CPL>(mp.hl, mp.sub, mp.LPH, j);
    const int key0 = (d - r) / 8;
    // Sliced keys: every warp scores its own value heads from their key
    // slices, the LPH lanes of a head taking its ckh key chunks in turn, so no
    // warp carries the others' key work and no score crosses warps. (Before,
    // the warps owning the tail scored every head and staged every key-path
    // term: one block barrier more per item, a third of the block idle at
    // each, and 255 registers: low-rank block backward 18.89 -> 18.75 ms with
    // three stages, 18.44 ms with two and three blocks per SM.) A lane holds
    // r/1024 key chunks, rounded up: the four-warp shapes have r = d/4 or d/2
    // (coop_supported), so at most half of CPL (KM slots).
    constexpr int KM = LR ? (CPL + 1) / 2 : CPL;
    const int ckh = r / 8 / H;
    int kidx[KM];
    bool kval[KM];
#pragma unroll
    for (int u = 0; u < KM; ++u) {
        kval[u] = !LR || mp.sub + mp.LPH * u < ckh;
        kidx[u] = LR ? key0 + mp.h * ckh + mp.sub + mp.LPH * u : cidx[u];
    }
    float qg[KM][8], U[KM][8];
    const float inv_width = 1.0f / (float)(a.norm_full ? d : r);

    const int64_t GB = gridDim.x, gb = blockIdx.x;
    // tokens gb, gb + GB, ..., every source of each in list order: at any
    // time the blocks read neighbouring tokens of the same row
    const int64_t ntok = gb < TT ? (TT - 1 - gb) / GB + 1 : 0;
    const int64_t lo = 0, hi = ntok * N;
    const uint64_t pol = l2_policy_evict_first();

    int64_t issued = lo, tok_p = gb;
    int n_p = 0, slot_p = 0;
    auto issue_next = [&]() {
        if (threadIdx.x == 0) {
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
        if (++n_p == N) { n_p = 0; tok_p += GB; }
        if (++slot_p == S) slot_p = 0;
    };
    for (int s = 0; s < S && issued < hi; ++s) issue_next();
    // q*g after the first copies are issued, so that their latency starts at
    // once (delta 8B backward phase 19.50 -> 19.42 ms)
#pragma unroll
    for (int j = 0; j < KM; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = kidx[j] * 8 + (e ^ sw) - key0 * 8;
            qg[j][e] = kval[j] ? ldg_chk(a.q + c * a.q_stride) * (a.g ? ldg_chk(a.g + c * a.g_stride) : 1.0f) : 0.f;
            U[j][e] = 0.f;
        }

    auto fetch_token = [&](int64_t t) {   // this thread's chunks, in 16-byte pieces
        const T *grow = static_cast<const T *>(a.dout) + t * d;
        const T *orow = static_cast<const T *>(a.fout) + t * d;
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int k = 0; k < CB / 16; ++k) {
                const int off = cidx[j] * 8 + k * (16 / (int)sizeof(T));
                cp_async16(tbuf + off, grow + off);
                cp_async16(tbuf + d + off, orow + off);
            }
        cp_async_commit();
    };
    if (kTok && hi > lo) fetch_token(gb);

    float G[CPL][8];
    float S_h = 0.f, lse_h = 0.f, dal = 0.f;
    const float alpha = a.alpha ? ldg_chk(a.alpha) : 1.0f;
    int64_t tok = gb, i = lo;
    int n = 0, slot = 0, par = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (; i < hi; ++i) {
        if (i == lo || n == 0) {
            const T *grow = static_cast<const T *>(a.dout) + tok * d;
            const T *orow = static_cast<const T *>(a.fout) + tok * d;
            if (!kTok && threadIdx.x == 0 && tok + GB < TT) {  // next token's rows, into L2
                prefetch_l2(grow + GB * d, vbytes);
                prefetch_l2(orow + GB * d, vbytes);
            }
            if (kTok) cp_async_wait_all();
            float sp = 0.f, raw = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                float o[8];
                if (kTok) {
                    ld_chunk_s_sw(tbuf + cidx[j] * 8, sw, G[j]);
                    ld_chunk_s_sw(tbuf + d + cidx[j] * 8, sw, o);
                } else {
                    ld_chunk_g_sw(grow + cidx[j] * 8, sw, G[j]);
                    ld_chunk_g_sw(orow + cidx[j] * 8, sw, o);
                }
                if (a.dalpha) raw = __fadd_rn(raw, dot8(G[j], o));
                if (a.alpha) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) G[j][e] *= alpha;  // delta form: G = alpha dL/dh
                }
                sp = __fadd_rn(sp, dot8(G[j], o));
            }
            S_h = a.coupling ? ldg_chk(a.coupling + (tok * H + mp.h)) : group_sum(sp, mp.LPH);
            if (kTok && tok + GB < TT) fetch_token(tok + GB);   // this thread's chunks are read
            if (a.dalpha && n == 0) dal += warp_sum(raw);  // each token counted once
            lse_h = ldg_chk(a.lse + tok * H + mp.h);
        }
        // the source's inverse RMS (a small, cache-resident table), requested
        // before the wait for the staged row so that its latency hides there
        const float iv = ldg_chk(a.inv + tok * a.inv_ld + s_rows[n]);
        // The first block barrier of an item also carries the wait's outcome
        // (all threads leave together on a timeout); with sliced keys it also
        // frees the stage of the previous item, which every warp has finished
        // by then.
        const bool got = mbar_wait(&bars[slot], (phase >> slot) & 1u, kWaitLimit);
        unsigned char *vb = ring + (size_t)slot * slot_bytes;
        float *gb_s = reinterpret_cast<float *>(vb + vbytes);
        const bool first = (s_first[n >> 5] >> (n & 31)) & 1u;

        // pass A: value dots, raw scores (full keys: over the value chunks;
        // sliced keys: over this lane's key chunks of its head's key slice)
        float v[CPL][8];
        float P = 0.f, zr = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            ld_chunk_s_sw(reinterpret_cast<const T *>(vb + cidx[j] * CB), sw, v[j]);
            P = __fadd_rn(P, dot8(G[j], v[j]));
            if constexpr (!LR) zr = __fadd_rn(zr, dot8(qg[j], v[j]));
        }
        if constexpr (LR) {
#pragma unroll
            for (int u = 0; u < KM; ++u)
                if (kval[u]) {
                    float kv[8];
                    ld_chunk_s_sw(reinterpret_cast<const T *>(vb + kidx[u] * CB), sw, kv);
                    zr = __fadd_rn(zr, dot8(qg[u], kv));
                }
        }
        P = group_sum(P, mp.LPH);
        zr = group_sum(zr, mp.LPH);
        const float wgt = exp2f((__fmul_rn(iv, zr) - lse_h) * kLog2e);
        const float dz = wgt * (P - S_h);
        const float cpart = warp_sum(mp.sub == 0 ? dz * zr : 0.f);
        if (lane == 0) cws[par * 32 + w] = cpart;
        // the item's one block barrier: the coupling sums, and the stage
        // wait's outcome (all threads leave together on a timeout); every
        // warp is past the previous item, whose stage thread 0 refills now
        // (full keys refilled it at once behind a second barrier at the end
        // of each item before: delta 8B backward 19.50 -> 18.51 ms)
        if (__syncthreads_or(!got)) { ok = false; break; }
        phase ^= 1u << slot;
        if (i > lo && issued < hi) issue_next();
        float C = 0.f;
#pragma unroll
        for (int k = 0; k < kCoopWarps; ++k) C += cws[par * 32 + k];
        const float coef = iv * iv * iv * C * inv_width;
        float *grad_row = a.grad + ((int64_t)s_rows[n] * TT + tok) * d;
        const float ak = iv * dz;

        if constexpr (!LR) {
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                float nv[8];
                if (first) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) nv[e] = 0.f;
                } else {
                    ld_chunk_s_sw(gb_s + cidx[j] * 8, sw, nv);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    nv[e] = fmaf(wgt, G[j][e], nv[e]);
                    nv[e] = fmaf(ak, qg[j][e], nv[e]);
                    nv[e] = fmaf(-coef, v[j][e], nv[e]);
                    U[j][e] = fmaf(ak, v[j][e], U[j][e]);
                }
                st_grad8(grad_row + cidx[j] * 8, sw, nv, a.grad_v8);
            }
        } else {
            // key-path terms of this lane's key chunks, staged in the shared
            // gradient row (the tail belongs to the last warps' value columns)
#pragma unroll
            for (int u = 0; u < KM; ++u)
                if (kval[u]) {
                    float kv[8], nv[8];
                    ld_chunk_s_sw(reinterpret_cast<const T *>(vb + kidx[u] * CB), sw, kv);
                    if (first) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) nv[e] = 0.f;
                    } else {
                        ld_chunk_s_sw(gb_s + kidx[u] * 8, sw, nv);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        nv[e] = fmaf(ak, qg[u][e], nv[e]);
                        nv[e] = fmaf(-coef, kv[e], nv[e]);
                        U[u][e] = fmaf(ak, kv[e], U[u][e]);
                    }
                    float *dst = gb_s + kidx[u] * 8;
                    AR_GUARD_S(dst, 32, 16, continue)
                    *reinterpret_cast<float4 *>(dst + sw) = make_float4(nv[0], nv[1], nv[2], nv[3]);
                    *reinterpret_cast<float4 *>(dst + (sw ^ 4)) = make_float4(nv[4], nv[5], nv[6], nv[7]);
                }
            // the warps owning tail columns wait for every warp's key-path
            // terms; the others only signal theirs (named barrier 1)
            if (mp.key_warp) bar_sync_named(1, kCoopWarps * 32);
            else bar_arrive_named(1, kCoopWarps * 32);
            // value path (and the radial term off the slice for the full norm)
            const float cv = a.norm_full ? coef : 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const bool tail = cidx[j] >= key0;
                float nv[8];
                if (tail || !first) {
                    ld_chunk_s_sw(gb_s + cidx[j] * 8, sw, nv);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) nv[e] = 0.f;
                }
                const float c2 = tail ? 0.f : cv;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    nv[e] = fmaf(wgt, G[j][e], nv[e]);
                    nv[e] = fmaf(-c2, v[j][e], nv[e]);
                }
                st_grad8(grad_row + cidx[j] * 8, sw, nv, a.grad_v8);
            }
        }
        par ^= 1;
        if (++n == N) { n = 0; tok += GB; }
        if (++slot == S) slot = 0;
    }
    if (!ok) {
        if (threadIdx.x == 0) {
            report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
            for (int64_t j = i; j < issued; ++j) {
                mbar_wait(&bars[slot], (phase >> slot) & 1u, kDrainLimit);
                phase ^= 1u << slot;
                if (++slot == S) slot = 0;
            }
        }
    }
    // per-block partial sums U over the key coordinates -> workspace row gb;
    // dL/dalpha partials (one per warp) -> tail
    {
        float *wrow = a.ws + gb * r;
#pragma unroll
        for (int j = 0; j < KM; ++j)
            if (kval[j]) st_f32x8_g_sw(wrow + (kidx[j] - key0) * 8, sw, U[j]);
    }
    if (a.dalpha && lane == 0) st_chk(a.ws + (GB * r + gb * 4 + w), dal);
}

template <typename T, int CPL, bool LR, bool FRESH>
cudaError_t coop_fwd_inst2(const RouteArgs &a, cudaStream_t s)
{
    const void *k = reinterpret_cast<const void *>(&route_fwd_coop_kernel<T, CPL, LR, FRESH>);
    const size_t smem = coop_fwd_smem_bytes(a.d, sizeof(T),
                                            a.partial != nullptr || (a.fresh1 && a.acc_row >= 0));
    int grid = 0;
    cudaError_t e = persistent_grid(k, kCoopWarps * 32, smem, &grid);
    if (e != cudaSuccess) return e;
    route_fwd_coop_kernel<T, CPL, LR, FRESH><<<grid, kCoopWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

// The fused-append variant when the host asks for it (fresh1).
template <typename T, int CPL, bool LR>
cudaError_t coop_fwd_inst(const RouteArgs &a, cudaStream_t s)
{
    return a.fresh1 ? coop_fwd_inst2<T, CPL, LR, true>(a, s) : coop_fwd_inst2<T, CPL, LR, false>(a, s);
}

template <typename T, int CPL, bool LR>
cudaError_t coop_bwd_inst(const RouteArgs *a, cudaStream_t s, int *grid_rows)
{
    const void *k = reinterpret_cast<const void *>(&route_bwd_coop_kernel<T, CPL, LR>);
    const size_t smem = coop_bwd_smem_bytes(a->d, sizeof(T), LR);
    int grid = 0;
    cudaError_t e = persistent_grid(k, kCoopWarps * 32, smem, &grid);
    if (e != cudaSuccess) return e;
    if (grid_rows) {
        *grid_rows = grid;
        return cudaSuccess;
    }
    route_bwd_coop_kernel<T, CPL, LR><<<grid, kCoopWarps * 32, smem, s>>>(*a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_coop_fwd(const RouteArgs &a, cudaStream_t s)
{
    const bool lr = a.r < a.d;
#define AR_COOP_CASE(C) \
    case C: return lr ? coop_fwd_inst<T, C, true>(a, s) : coop_fwd_inst<T, C, false>(a, s);
    switch (a.d / 1024) {
        AR_COOP_CASE(1) AR_COOP_CASE(2) AR_COOP_CASE(3) AR_COOP_CASE(4)
        AR_COOP_CASE(5) AR_COOP_CASE(6) AR_COOP_CASE(7) AR_COOP_CASE(8)
    default: return cudaErrorNotSupported;
    }
#undef AR_COOP_CASE
}

template <typename T>
cudaError_t dispatch_coop_bwd(const RouteArgs *a, cudaStream_t s, int *grid_rows)
{
    const bool lr = a->r < a->d;
#define AR_COOP_CASE(C)                                                   \
    case C:                                                               \
        return lr ? coop_bwd_inst<T, C, true>(a, s, grid_rows)            \
                  : coop_bwd_inst<T, C, false>(a, s, grid_rows);
    switch (a->d / 1024) {
        AR_COOP_CASE(1) AR_COOP_CASE(2) AR_COOP_CASE(3) AR_COOP_CASE(4)
        AR_COOP_CASE(5) AR_COOP_CASE(6) AR_COOP_CASE(7) AR_COOP_CASE(8)
    default: return cudaErrorNotSupported;
    }
#undef AR_COOP_CASE
}

}  // namespace ar

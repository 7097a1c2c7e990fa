// Fused routing backward for sm_103a, full-width keys (r = d).
//
// For one routing site, given dL/dout, emits dL/ds_n for every listed source
// into the shared fp32 gradient rows (store on a row's first touch, in-place
// accumulation afterwards: "Multi-Head Attention Residuals", Appendix E,
// Figure 10) and per-block partial sums for dL/dq and dL/dg.
//
// Per token t, source n, head h (w = softmax weight, recomputed from the
// saved log-sum-exp; G = dL/dout):
//   P[n,h]   = <G_[h], s_{n,[h]}>
//   zr[n,h]  = sum_{c in slice h} q_c g_c s_{n,c}       (z = inv_n * zr)
//   S[h]     = sum_n w P = <G_[h], out_[h]>  (the softmax coupling term, read
//              from the forward output instead of a second pass over the
//              sources: out_[h] is exactly sum_n w s_{n,[h]})
//   dz[n,h]  = w (P - S)                      (routing feedback,
//              "Low-Rank Attention Residuals", Eq. 15 / Lemma 2)
//   dL/ds_n  = w G + inv dz (q g)   on slice h
//            - inv^3 / d * (sum_h dz zr) * s_n   on all coordinates
//              (score gradient through the RMS: MHAR Appendix E, LR-AttnRes
//              Eq. 21 with r = d)
//   dq_c = g_c U_c, dg_c = q_c U_c with U_c = sum_{t,n} inv dz s_{n,c}.
// Every (token, source) item is independent once S[h] and lse[h] are known.
// Warp w takes tokens w, w + W, ... (W warps in the grid) and every source of
// each in list order, so at any time the warps read neighbouring tokens of
// the same rows. (An equal contiguous range of the T*N items per warp splits
// the work exactly, but then neighbouring warps sit on different rows: 1B
// backward 91.35 -> 90.42 ms with the strided order.)
//
// GB300 mapping: one warp per item stream with a private ring of
// shared-memory stages, as in the forward; a stage holds the source row
// (storage dtype) and, unless this is the row's first touch, its fp32
// gradient row, both brought in by 1-D bulk copies on one mbarrier. The new
// gradient row goes back with one 256-bit store per 8-element chunk (a whole
// 32-byte sector; two 16-byte stores for rows of four chunks per lane or
// fewer, or a gradient base that is not 32-byte aligned). G, q*g, U and the staged row's
// values stay in registers (8*CPL floats each). Lanes whose bit 2 is set keep
// each chunk's two halves swapped, so that their 16-byte reads of the fp32
// gradient row fall on the other half of the banks; dot products are summed
// as (low half) + (high half), which gives the forward's bits either way.
#pragma once

#include "common.cuh"
#include "launch_util.cuh"

namespace ar {

constexpr int kBwdWarps = 4;
// Two stages of (source row + fp32 gradient row) per warp, plus a per-warp
// buffer into which each lane fetches its own chunks of the next token's
// dL/dout and forward-output rows by cp.async while the current token's items
// run, so a token's first item does not wait on DRAM for them. Against three
// stages and plain loads of the token rows: 1B backward phase 90.54 -> 89.65
// ms, 350M 33.13 -> 32.53 ms, 100M 4.63 -> 4.53 ms (three stages with the
// buffer were slower on 512-wide rows).
constexpr int kBwdStages = 2;

inline size_t bwd_smem_bytes(int d, size_t esize)
{
    return (size_t)kBwdWarps * kBwdStages * ((size_t)d * esize + (size_t)d * 4) +
           (size_t)kBwdWarps * kBwdStages * 8 + (size_t)kBwdWarps * AR_MAX_SOURCES * 4 +
           (size_t)kBwdWarps * 2 * d * esize;
}

// CS: the coupling term comes from a.coupling (ar_route_bwd_exact), not from
// the forward output (a separate instantiation keeps the one-pass kernel as
// it was)
template <typename T, int CPL, bool CS = false>
__global__ void __launch_bounds__(kBwdWarps * 32, CPL <= 2 ? 4 : 1)
    route_bwd_kernel(const __grid_constant__ RouteArgs a)
{
    AR_CHK_ENTER(a);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    __shared__ uint32_t s_first[AR_MAX_SOURCES / 32];
    constexpr int S = kBwdStages;
    constexpr int CB = ChunkBytes<T>::value;
    constexpr unsigned FULL = 0xffffffffu;
    // 256-bit gradient stores: measured faster from five chunks per lane up
    // (1B shape: 8 heads -2 %, 16 heads -8 %), slightly slower below (the
    // lane-order selects cost more than the halved store count saves)
    constexpr bool kV8 = CPL >= 5;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, N = a.n_src, H = a.H;
    const int64_t TT = a.T;
    const uint32_t vbytes = (uint32_t)d * (uint32_t)sizeof(T);
    const uint32_t gbytes = (uint32_t)d * 4u;
    const uint32_t slot_bytes = vbytes + gbytes;

    unsigned char *rings = smem;
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + (size_t)kBwdWarps * S * slot_bytes);
    float *inv_all = reinterpret_cast<float *>(bars_all + kBwdWarps * S);

    for (int i = threadIdx.x; i < N; i += blockDim.x) s_rows[i] = a.rows[i];
    for (int i = threadIdx.x; i < AR_MAX_SOURCES / 32; i += blockDim.x) s_first[i] = a.first_mask[i];
    unsigned char *ring = rings + (size_t)warp * S * slot_bytes;
    uint64_t *bars = bars_all + warp * S;
    float *cur_inv = inv_all + warp * AR_MAX_SOURCES;
    // this warp's token buffer: the next token's dL/dout row, then its output
    // row, fetched by each lane for its own chunks while the current token runs
    T *tbuf = reinterpret_cast<T *>(inv_all + kBwdWarps * AR_MAX_SOURCES) + (size_t)warp * 2 * d;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // ---- lane -> head and chunk mapping (same chunks as the forward); lanes
    // with sw = 4 keep their chunks' halves swapped (conflict-free fp32 reads)
    const int LPH = 32 / H;
    const int h = lane / LPH, sub = lane - h * LPH;
    const int sw = ((lane >> 2) & 1) * 4;
    int cidx[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) cidx[j] = chunk_of<CPL>(h, sub, LPH, j);
    // q*g of this lane's chunks; on rows of up to 512 columns loaded after the
    // first copies are issued, so that their latency starts at once (100M
    // backward phase 4.500 -> 4.482 ms; on wider rows it measured no faster)
    constexpr bool kQgLate = CPL <= 2;
    float qg[CPL][8];
    auto load_qg = [&]() {
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int c = cidx[j] * 8 + (e ^ sw);
                qg[j][e] = ldg_chk(a.q + c * a.q_stride) * (a.g ? ldg_chk(a.g + c * a.g_stride) : 1.0f);
            }
    };
    if constexpr (!kQgLate) load_qg();
    const float inv_d = 1.0f / (float)d;

    // ---- this warp's tokens gw, gw + GW, ..., every source of each in list
    // order: at any time the warps read neighbouring tokens of the same row
    const int64_t GW = (int64_t)gridDim.x * kBwdWarps;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + warp;
    const int64_t ntok = gw < TT ? (TT - 1 - gw) / GW + 1 : 0;
    const int64_t lo = 0, hi = ntok * N;
    const uint64_t pol = l2_policy_evict_first();

    int64_t issued = lo, tok_p = gw;
    int n_p = 0, slot_p = 0;
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
        if (++n_p == N) { n_p = 0; tok_p += GW; }
        if (++slot_p == S) slot_p = 0;
    };
    for (int s = 0; s < S && issued < hi; ++s) issue_next();
    if constexpr (kQgLate) load_qg();

    float U[CPL][8];
#pragma unroll
    for (int j = 0; j < CPL; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) U[j][e] = 0.f;

    constexpr int kPieces = CB / 16;   // 16-byte pieces per chunk
    auto fetch_token = [&](int64_t t) {
        const T *grow = static_cast<const T *>(a.dout) + t * d;
        const T *orow = static_cast<const T *>(a.fout) + t * d;
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int k = 0; k < kPieces; ++k) {
                const int off = cidx[j] * 8 + k * (16 / (int)sizeof(T));
                cp_async16(tbuf + off, grow + off);
                cp_async16(tbuf + d + off, orow + off);
            }
        cp_async_commit();
    };
    if (hi > lo) fetch_token(gw);

    float G[CPL][8];
    float S_h = 0.f, lse_h = 0.f, dal = 0.f;
    const float alpha = a.alpha ? ldg_chk(a.alpha) : 1.0f;
    int64_t tok = gw, i = lo;
    int n = 0, slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (; i < hi; ++i) {
        if (i == lo || n == 0) {
            // token-level data: dL/dout, the coupling term S, lse, inverse RMS
            cp_async_wait_all();
            float sp = 0.f, raw = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                float o[8];
                ld_chunk_s_sw(tbuf + cidx[j] * 8, sw, G[j]);
                ld_chunk_s_sw(tbuf + d + cidx[j] * 8, sw, o);
                if (a.dalpha) raw = __fadd_rn(raw, dot8(G[j], o));
                if (a.alpha) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) G[j][e] *= alpha;  // delta form: G = alpha dL/dh
                }
                sp = __fadd_rn(sp, dot8(G[j], o));
            }
            if constexpr (CS) S_h = ldg_chk(a.coupling + (tok * H + h));
            else S_h = group_sum(sp, LPH);
            if (tok + GW < TT) fetch_token(tok + GW);      // this lane's chunks are read
            if (a.dalpha && n == 0) dal += warp_sum(raw);  // each token counted by the warp owning (t, 0)
            lse_h = ldg_chk(a.lse + tok * H + h);
            __syncwarp();
            for (int nn = lane; nn < N; nn += 32)
                cur_inv[nn] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[nn]);
            __syncwarp();
        }
        const bool got = mbar_wait(&bars[slot], (phase >> slot) & 1u, kWaitLimit);
        if (!__all_sync(FULL, got)) { ok = false; break; }
        phase ^= 1u << slot;
        const unsigned char *vb = ring + (size_t)slot * slot_bytes;
        const float *gb = reinterpret_cast<const float *>(vb + vbytes);
        const bool first = (s_first[n >> 5] >> (n & 31)) & 1u;

        // pass 1: value dot with G and raw score (the forward's sum order)
        float v[CPL][8];
        float P = 0.f, zr = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            ld_chunk_s_sw(reinterpret_cast<const T *>(vb + cidx[j] * CB), sw, v[j]);
            P = __fadd_rn(P, dot8(G[j], v[j]));
            zr = __fadd_rn(zr, dot8(qg[j], v[j]));
        }
        P = group_sum(P, LPH);
        zr = group_sum(zr, LPH);
        const float iv = cur_inv[n];
        const float w = exp2f((__fmul_rn(iv, zr) - lse_h) * kLog2e);
        const float dz = w * (P - S_h);
        const float C = (H == 1) ? dz * zr : warp_sum(sub == 0 ? dz * zr : 0.f);
        const float coef = iv * iv * iv * C * inv_d;
        const float ak = iv * dz;
        float *grad_row = a.grad + ((int64_t)s_rows[n] * TT + tok) * d;

        // pass 2: gradient row
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            float nv[8];
            if (first) {
#pragma unroll
                for (int e = 0; e < 8; ++e) nv[e] = 0.f;
            } else {
                ld_chunk_s_sw(gb + cidx[j] * 8, sw, nv);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                nv[e] = fmaf(w, G[j][e], nv[e]);
                nv[e] = fmaf(ak, qg[j][e], nv[e]);
                nv[e] = fmaf(-coef, v[j][e], nv[e]);
                U[j][e] = fmaf(ak, v[j][e], U[j][e]);
            }
            st_grad8(grad_row + cidx[j] * 8, sw, nv, kV8 && a.grad_v8);
        }
        __syncwarp();
        if (issued < hi) issue_next();
        if (++n == N) { n = 0; tok += GW; }
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

    // The block's partial sums: each warp puts U in its own (now idle) part of
    // the ring, then the block adds the warps in order into workspace row
    // blockIdx.x (a quarter of the rows a per-warp layout would leave for
    // the reduction to read); dL/dalpha partials -> tail.
    __syncthreads();
    float *uw = reinterpret_cast<float *>(ring);
#pragma unroll
    for (int j = 0; j < CPL; ++j) st_f32x8_s_sw(uw + cidx[j] * 8, sw, U[j]);
    __shared__ float s_dal[kBwdWarps];
    if (lane == 0) s_dal[warp] = dal;
    __syncthreads();
    const int64_t GB = gridDim.x, gb = blockIdx.x;
    const size_t wstride = (size_t)S * slot_bytes / sizeof(float);
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < kBwdWarps; ++k) t += reinterpret_cast<const float *>(rings)[k * wstride + c];
        st_chk(a.ws + (gb * d + c), t);
    }
    if (a.dalpha && threadIdx.x == 0) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < kBwdWarps; ++k) t += s_dal[k];
        AR_GUARD_G(a.ws + GB * d + gb * 4, 16, true, 16, return)
        *reinterpret_cast<float4 *>(a.ws + GB * d + gb * 4) = make_float4(t, 0.f, 0.f, 0.f);
    }
}

template <typename T, int CPL, bool CS>
cudaError_t bwd_inst_cs(const RouteArgs *a, cudaStream_t s, int *grid_rows)
{
    const void *k = reinterpret_cast<const void *>(&route_bwd_kernel<T, CPL, CS>);
    const size_t smem = bwd_smem_bytes(a->d, sizeof(T));
    int grid = 0;
    cudaError_t e = persistent_grid(k, kBwdWarps * 32, smem, &grid);
    if (e != cudaSuccess) return e;
    if (grid_rows) {
        *grid_rows = grid;  // workspace rows: one per block
        return cudaSuccess;
    }
    route_bwd_kernel<T, CPL, CS><<<grid, kBwdWarps * 32, smem, s>>>(*a);
    return cudaGetLastError();
}

template <typename T, int CPL>
cudaError_t bwd_inst(const RouteArgs *a, cudaStream_t s, int *grid_rows)
{
    return a->coupling ? bwd_inst_cs<T, CPL, true>(a, s, grid_rows)
                       : bwd_inst_cs<T, CPL, false>(a, s, grid_rows);
}

// Same shapes as the forward. With grid_rows != nullptr only the grid (in
// blocks = workspace rows) is computed and nothing is launched.
template <typename T>
cudaError_t dispatch_bwd(const RouteArgs *a, cudaStream_t s, int *grid_rows)
{
    if (a->r != a->d) return cudaErrorNotSupported;
    switch (a->d / 256) {
    case 1: return bwd_inst<T, 1>(a, s, grid_rows);
    case 2: return bwd_inst<T, 2>(a, s, grid_rows);
    case 3: return bwd_inst<T, 3>(a, s, grid_rows);
    case 4: return bwd_inst<T, 4>(a, s, grid_rows);
    case 5: return bwd_inst<T, 5>(a, s, grid_rows);
    case 6: return bwd_inst<T, 6>(a, s, grid_rows);
    case 7: return bwd_inst<T, 7>(a, s, grid_rows);
    case 8: return bwd_inst<T, 8>(a, s, grid_rows);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace ar

// Multi-query forward: the reads of several sites over one source list, in one
// pass over the sources ("Low-Rank Attention Residuals", Sec. 3.4: with
// input-independent queries, the inter-block reads of every site of a block
// can be done first, together, and each site's intra-block read merged in
// later by the online-softmax update).
//
// For queries q_1..q_nq (each with its norm weight g_i) and one row list,
// every token gets nq outputs out_i = sum_n softmax_n(z_i[n, h]) s_n on each
// head's value slice, and nq log-sum-exps, as nq calls of the single-query
// forward would give; the rows are read once instead of nq times.
//
// One block of 256 threads per token at a time (persistent over tokens). All
// N rows of a token are staged together (N bulk copies on one mbarrier, two
// token buffers, so the next token's rows arrive during this one's work):
//   1. scores: thread k owns key chunk k (8 key columns) for the whole kernel
//      and keeps q_i*g_i of its chunk for every query in registers; for each
//      row and query it forms the chunk's partial score, sums it over the
//      aligned lanes of its key slice in the warp, and publishes one piece;
//   2. softmax: one thread per (query, head) adds the pieces of each row in
//      order, scales by the row's inverse RMS (adding log k for a row listed k
//      times), and writes the normalised weights and the lse;
//   3. mix: thread t takes chunks t, t + 256, ...; per chunk it sums the N
//      staged rows with each query's weights (nq accumulators of 8) and
//      stores the nq output chunks.
// Three block barriers per token.
#pragma once

#include "common.cuh"
#include "launch_util.cuh"

namespace ar {

constexpr int kMultiThreads = 256;

// Lanes whose partial scores are summed in-warp: the largest power of two up
// to 32 that divides a key slice's chunk count, so the groups are aligned and
// never straddle slices; a slice is then added up from its pieces.
__host__ __device__ inline int multi_kg(int r, int H)
{
    const int kch = r / H / 8;
    int kg = 32;
    while (kg > 1 && kch % kg != 0) kg >>= 1;
    return kg;
}

// Token buffers that fit (2, or 1), or 0 when even one does not.
inline int multi_fwd_buffers(int d, int r, int H, int N, int nq, size_t esize, size_t *smem)
{
    const size_t fixed = 2 * 8                                            // mbarriers
                         + (size_t)nq * N * (r / 8 / multi_kg(r, H)) * 4  // score pieces
                         + (size_t)nq * H * N * 4                         // weights
                         + (size_t)N * 4;                                 // inverse RMS
    const size_t tok = (size_t)N * d * esize;
    for (int nb = 2; nb >= 1; --nb)
        if (nb * tok + fixed <= 200 * 1024) {
            *smem = nb * tok + fixed;
            return nb;
        }
    return 0;
}

template <typename T>
__global__ void __launch_bounds__(kMultiThreads)
    route_fwd_multi_kernel(const __grid_constant__ MultiArgs m, int nbuf)
{
    AR_CHK_ENTER(m.base);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[AR_MAX_SOURCES];
    constexpr int CB = ChunkBytes<T>::value;
    constexpr int QM = AR_MAX_QUERIES;
    const RouteArgs &a = m.base;
    const int tid = threadIdx.x;
    const int d = a.d, r = a.r, N = a.n_src, H = a.H, nq = m.nq;
    const int64_t TT = a.T;
    const uint32_t row_bytes = (uint32_t)d * (uint32_t)sizeof(T);
    const uint32_t tok_bytes = (uint32_t)N * row_bytes;
    const int K = d / H, kch = r / H / 8, key0 = (d - r) / 8, nch = d / 8;
    const int kg = multi_kg(r, H), ppk = kch / kg, pieces = r / 8 / kg;

    for (int i = tid; i < N; i += kMultiThreads) s_rows[i] = a.rows[i];
    unsigned char *bufs = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(bufs + (size_t)nbuf * tok_bytes);
    float *zpc = reinterpret_cast<float *>(bars + 2);        // [nq][N][pieces]
    float *wts = zpc + (size_t)nq * N * pieces;               // [nq][H][N]
    float *invs = wts + (size_t)nq * H * N;                   // [N]
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }

    // this thread's key chunk (if any) and its q*g for every query
    const int kc = tid;
    const bool has_key = kc < r / 8;
    const bool key_warp = (tid & ~31) < r / 8;    // warp holds key chunks: joins the shuffles
    float qg[QM][8];
#pragma unroll
    for (int qi = 0; qi < QM; ++qi)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = kc * 8 + e;
            qg[qi][e] = (has_key && qi < nq)
                            ? ldg_chk(m.q[qi] + c) * (m.g[qi] ? ldg_chk(m.g[qi] + c) : 1.0f)
                            : 0.f;
        }
    __syncthreads();

    const int64_t GB = gridDim.x, gb = blockIdx.x;
    const uint64_t pol = l2_policy_evict_first();
    auto issue_token = [&](int64_t tok, int b) {  // thread 0: all N rows of a token
        unsigned char *dst = bufs + (size_t)b * tok_bytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[b], tok_bytes);
        for (int n = 0; n < N; ++n)
            bulk_g2s(dst + (size_t)n * row_bytes,
                     static_cast<const unsigned char *>(a.bank) +
                         ((int64_t)s_rows[n] * TT + tok) * row_bytes,
                     row_bytes, &bars[b], pol);
    };
    if (tid == 0) {
        for (int b = 0; b < nbuf; ++b)
            if (gb + b * GB < TT) issue_token(gb + b * GB, b);
    }

    uint32_t phase = 0;
    int b = 0;
    bool ok = true;
    for (int64_t tok = gb; tok < TT; tok += GB) {
        for (int n = tid; n < N; n += kMultiThreads)
            invs[n] = ldg_chk(a.inv + tok * a.inv_ld + s_rows[n]);
        const bool got = mbar_wait(&bars[b], (phase >> b) & 1u, kWaitLimit);
        const unsigned char *buf = bufs + (size_t)b * tok_bytes;

        // 1. score pieces
        if (key_warp) {
            for (int n = 0; n < N; ++n) {
                float kv[8];
                ld_chunk_s(reinterpret_cast<const T *>(buf + (size_t)n * row_bytes +
                                                       (size_t)(key0 + (has_key ? kc : 0)) * CB),
                           kv);
#pragma unroll
                for (int qi = 0; qi < QM; ++qi) {
                    if (qi >= nq) continue;
                    float zp = has_key ? dot8(qg[qi], kv) : 0.f;
                    zp = group_sum(zp, kg);
                    if (has_key && (kc % kg) == 0) zpc[((size_t)qi * N + n) * pieces + kc / kg] = zp;
                }
            }
        }
        if (__syncthreads_or(!got)) { ok = false; break; }
        phase ^= 1u << b;

        // 2. weights and lse per (query, head)
        for (int p = tid; p < nq * H; p += kMultiThreads) {
            const int qi = p / H, hh = p - qi * H;
            float *wq = wts + (size_t)p * N;
            float mx = 0.f;
            for (int n = 0; n < N; ++n) {
                const float *pc = zpc + ((size_t)qi * N + n) * pieces + hh * ppk;
                float zr = 0.f;
                for (int k = 0; k < ppk; ++k) zr += pc[k];
                float z = __fmul_rn(zr, invs[n]);
                if (a.has_bias) z = __fadd_rn(z, a.bias[n]);
                wq[n] = z;
                mx = n == 0 ? z : fmaxf(mx, z);
            }
            float l = 0.f;
            for (int n = 0; n < N; ++n) l += exp2f((wq[n] - mx) * kLog2e);
            const float lse = mx + log2f(l) * kLn2;
            for (int n = 0; n < N; ++n) wq[n] = exp2f((wq[n] - lse) * kLog2e);
            st_chk(m.lse[qi] + (tok * H + hh), lse);
        }
        __syncthreads();

        // 3. mix: nq outputs per chunk
        for (int c = tid; c < nch; c += kMultiThreads) {
            const int h = (c * 8) / K;
            float acc[QM][8];
#pragma unroll
            for (int qi = 0; qi < QM; ++qi)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[qi][e] = 0.f;
            for (int n = 0; n < N; ++n) {
                float v[8];
                ld_chunk_s(reinterpret_cast<const T *>(buf + (size_t)n * row_bytes + (size_t)c * CB), v);
#pragma unroll
                for (int qi = 0; qi < QM; ++qi) {
                    if (qi >= nq) continue;
                    const float w = wts[((size_t)qi * H + h) * N + n];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[qi][e] = fmaf(w, v[e], acc[qi][e]);
                }
            }
#pragma unroll
            for (int qi = 0; qi < QM; ++qi)
                if (qi < nq) st_chunk_g(static_cast<T *>(m.out[qi]) + tok * d + c * 8, acc[qi]);
        }
        // every thread is done with this buffer: the token nbuf steps ahead
        // can land in it
        __syncthreads();
        if (tid == 0 && tok + nbuf * GB < TT) issue_token(tok + nbuf * GB, b);
        if (++b == nbuf) b = 0;
    }
    if (!ok && tid == 0) {
        report_error(a.err, AR_DEVERR_WAIT_TIMEOUT);
        // wait briefly for the copies still in flight, then leave
        for (int k = 0; k < nbuf; ++k) {
            mbar_wait(&bars[b], (phase >> b) & 1u, kDrainLimit);
            phase ^= 1u << b;
            if (++b == nbuf) b = 0;
        }
    }
}

template <typename T>
cudaError_t dispatch_fwd_multi(const MultiArgs &m, cudaStream_t s)
{
    const RouteArgs &a = m.base;
    if (a.r / 8 > kMultiThreads) return cudaErrorNotSupported;  // one key chunk per thread
    size_t smem = 0;
    const int nbuf = multi_fwd_buffers(a.d, a.r, a.H, a.n_src, m.nq, sizeof(T), &smem);
    if (nbuf == 0) return cudaErrorNotSupported;
    const void *k = reinterpret_cast<const void *>(&route_fwd_multi_kernel<T>);
    int grid = 0;
    cudaError_t e = persistent_grid(k, kMultiThreads, smem, &grid);
    if (e != cudaSuccess) return e;
    if (a.T < grid) grid = (int)a.T;
    route_fwd_multi_kernel<T><<<grid, kMultiThreads, smem, s>>>(m, nbuf);
    return cudaGetLastError();
}

}  // namespace ar

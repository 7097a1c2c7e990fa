// Shape rules of the routing kernel families, shared by the host-side checks
// and the launches: which family serves (d, r, H, n_src), and the shared-memory
// sizes those rules depend on.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "ar_internal.h"

namespace ar {

// ---- one-warp sliced-key family ------------------------------------------------
constexpr int kLrFwdStages = 4;
constexpr int kLrBwdStages = 2;
constexpr size_t kLrSmemLimit = 200 * 1024;

// Column-block width of the mixing sweep: the largest multiple of 8 columns,
// at most 1024, that divides both the non-key width d - r and the key width r
// (blocks never straddle the start of the key tail).
__host__ __device__ inline int lr_block_cols(int d, int r)
{
    int x = d - r, y = r;
    while (y) { const int t = x % y; x = y; y = t; }   // gcd(d - r, r) (= r when r = d)
    for (int c = 1024; c >= 8; c -= 8)
        if (x % c == 0) return c;
    return 8;
}

inline size_t lr_fwd_smem_bytes(int d, int r, int N, int H, size_t esize)
{
    const size_t cw = (size_t)lr_block_cols(d, r);
    return 2 * (size_t)N * r * esize            // key cache, double-buffered
           + (size_t)kLrFwdStages * cw * esize  // value ring
           + 2 * (size_t)N * H * 4              // scores, weights
           + (size_t)(2 + kLrFwdStages) * 8     // mbarriers
           + (size_t)AR_MAX_SOURCES * 4 * 2;    // inverse RMS (current, next)
}

// 8-column key chunks per lane, in units of 256 key columns.
__host__ __device__ inline int lr_kmax(int r) { return (r + 255) / 256; }

// ---- scalar-access family ----------------------------------------------------------
// Blocks of the backward per SM. Each block reduces its warps' dq/dg partial
// sums into one workspace row, so the workspace (SMs x this rows) does not
// depend on the source count, which sets the warps per block.
constexpr int kGenBlocksPerSm = 2;
constexpr size_t kGenSmemLimit = 200 * 1024;

// Per-warp shared floats of the forward: weights [N, H], lse [H], inverse RMS [N].
__host__ __device__ inline size_t gen_fwd_warp_floats(int N, int H) { return (size_t)N * H + H + N; }
// ... of the backward: weights and score gradients [N, H] each, coupling S [H],
// C and inverse RMS [N] each, dq/dg partials [r].
__host__ __device__ inline size_t gen_bwd_warp_floats(int N, int H, int r)
{
    return 2 * (size_t)N * H + H + 2 * (size_t)N + r;
}

// Warps per block: 4, or fewer when the per-warp arrays are large; 0 when even
// one warp does not fit (the block also holds q*g, r floats).
inline int gen_block_warps(size_t warp_floats, int r)
{
    for (int w = 4; w >= 1; w >>= 1)
        if (((size_t)r + w * warp_floats) * 4 <= kGenSmemLimit) return w;
    return 0;
}

// ---- family choice -------------------------------------------------------------------
// r = d <= 2048, H a power of two <= 32: one warp per token (kFull).
// d a multiple of 1024 (coop_supported): four warps share each row (kCoop).
// Other d <= 4096 with whole 8-column key chunks per head and the key cache
// within its limit: one warp per token, two sweeps (kSliced).
// Everything else: one warp per token with scalar accesses (kGeneric), as long
// as its per-warp arrays fit. So do sites that list a row more than once
// (`repeats`): only these kernels add the log-multiplicity to a score, which
// keeps that term out of the tiled kernels' inner loops.
enum class Family { kFull, kCoop, kSliced, kGeneric, kNone };

inline Family family_of(int d, int r, int H, int N, size_t esize, bool repeats)
{
    if (H < 1 || d <= 0 || r <= 0 || r > d || d % H != 0 || r % H != 0) return Family::kNone;
    if (N < 1 || N > AR_MAX_SOURCES) return Family::kNone;
    if (!repeats && d % 256 == 0 && r % 8 == 0) {
        const bool pow2_h = H <= 32 && (32 % H) == 0;
        if (r == d && d <= 2048 && pow2_h) return Family::kFull;
        if (r % 256 == 0 && coop_supported(d, r, H)) return Family::kCoop;
        if (d <= 4096 && pow2_h && (r / H) % 8 == 0 && lr_kmax(r) <= 16 &&
            lr_fwd_smem_bytes(d, r, N, H, esize) <= kLrSmemLimit)
            return Family::kSliced;
    }
    if (gen_block_warps(gen_fwd_warp_floats(N, H), r) > 0 &&
        gen_block_warps(gen_bwd_warp_floats(N, H, r), r) > 0)
        return Family::kGeneric;
    return Family::kNone;
}

}  // namespace ar

// Shared device helpers of the GB300 depth-routing kernels: argument block,
// PTX wrappers for mbarriers and 1-D bulk (TMA) copies, and 8-element chunk
// conversions between the storage dtype and fp32 registers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ar_internal.h"
#include "attnres.h"
#include "checks.h"

namespace ar {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Online-softmax rescale threshold (log2 units): the running maximum is only
// moved when a score exceeds it by more than this, so the exponentials stay
// below 2^8 and most sources skip the rescale of the accumulator.
constexpr float kRescaleTau = 8.0f;
// Suspend-time hint of one mbarrier poll, in ns: a waiting thread sleeps until
// the phase completes or this much time has passed, instead of coming back at
// once and spinning on the poll (1B forward phase 18.57 -> 18.39 ms; the
// length of the hint made no difference between 10 us and 1 ms).
constexpr uint32_t kPollSuspendNs = 10000;
// Bound on mbarrier polls before a wait is declared lost (no device trap):
// about 1.3 s when every poll sleeps its whole hint.
constexpr uint32_t kWaitLimit = 1u << 17;
// Bound on the polls per stage when, after a lost wait, a warp waits for its
// copies still in flight before it leaves.
constexpr uint32_t kDrainLimit = 1u << 12;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- range checks (checked build) ---------------------------------------------
// Built with AR_CHECKED, every global access the helpers below make is first
// checked against the buffers of the launch (the table the host puts in the
// arguments), and every staged shared-memory access against the block's
// dynamic shared memory, both for range and alignment. A refused access is
// not made: a load gives zeros, a store is dropped, a bulk copy completes its
// bytes on its mbarrier without copying. The first refusal is recorded and
// AR_DEVERR_BOUNDS is set in the error word; nothing traps. A kernel names
// its arguments at entry (chk_enter) or opts out (chk_off). Without
// AR_CHECKED the checks are the constant true and compile away.
#ifdef AR_CHECKED
static __shared__ const RouteArgs *chk_args_s;
extern __shared__ __align__(16) unsigned char chk_dyn_smem[];

__device__ __forceinline__ void chk_enter(const RouteArgs &a) { chk_args_s = a.chk.off ? nullptr : &a; }
__device__ __forceinline__ void chk_off() { chk_args_s = nullptr; }

enum : uint32_t { kChkLoad = 1, kChkStore = 2, kChkShared = 3 };

static __device__ __noinline__ void chk_record(const RouteArgs *a, uint64_t addr, uint32_t bytes,
                                        uint32_t kind)
{
    unsigned long long *f = a->chk.fault;
    if (f && atomicCAS(f, 0ull, 1ull) == 0ull) {
        f[1] = addr;
        f[2] = (static_cast<unsigned long long>(kind) << 32) | bytes;
        __threadfence();
    }
    if (a->err) atomicOr(a->err, AR_DEVERR_BOUNDS);
}

// The decision itself (chk_decide, checks.h) is shared with a host test.
static __device__ __noinline__ bool chk_global(const void *p, uint32_t bytes, bool store, uint32_t align)
{
    const RouteArgs *a = chk_args_s;
    if (!a) return true;
    const uint64_t x = reinterpret_cast<uint64_t>(p);
    if (chk_decide(*a, x, bytes, store, align)) return true;
    chk_record(a, x, bytes, store ? kChkStore : kChkLoad);
    return false;
}

static __device__ __noinline__ bool chk_shared(const void *p, uint32_t bytes, uint32_t align)
{
    const RouteArgs *a = chk_args_s;
    if (!a) return true;
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint32_t x = smem_u32(p), base = smem_u32(chk_dyn_smem);
    if (x >= base && x + bytes <= base + dyn && (x | bytes) % align == 0) return true;
    chk_record(a, x, bytes, kChkShared);
    return false;
}
#define AR_CHK_G(p, n, st, al) ::ar::chk_global((p), (n), (st), (al))
#define AR_CHK_S(p, n, al) ::ar::chk_shared((p), (n), (al))
// run the statement(s) after the check's arguments when the access is refused
#define AR_GUARD_G(p, n, st, al, ...) \
    if (!::ar::chk_global((p), (n), (st), (al))) { __VA_ARGS__; }
#define AR_GUARD_S(p, n, al, ...) \
    if (!::ar::chk_shared((p), (n), (al))) { __VA_ARGS__; }
#define AR_CHK_ENTER(a) ::ar::chk_enter(a)
#define AR_CHK_OFF() ::ar::chk_off()
// kernels without a RouteArgs parameter take the table as a last parameter
#define AR_CHK_PARAM , const __grid_constant__ ::ar::RouteArgs chk_args
#define AR_CHK_PASS(a) , (a)
#define AR_CHK_ENTER_PARAM() ::ar::chk_enter(chk_args)
#else
#define AR_CHK_G(p, n, st, al) true
#define AR_CHK_S(p, n, al) true
#define AR_GUARD_G(p, n, st, al, ...)
#define AR_GUARD_S(p, n, al, ...)
#define AR_CHK_ENTER(a) ((void)0)
#define AR_CHK_OFF() ((void)0)
#define AR_CHK_PARAM
#define AR_CHK_PASS(a)
#define AR_CHK_ENTER_PARAM() ((void)0)
#endif

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` on the mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy)
{
#ifdef AR_CHECKED
    if (!chk_global(src, bytes, false, 16) || !chk_shared(dst, bytes, 16)) {
        // refused: the bytes complete without a copy, so no wait runs out
        asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(
                         smem_u32(bar)),
                     "r"(bytes)
                     : "memory");
        return;
    }
#endif
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Ask L2 to fetch `bytes` (a multiple of 16) from a 16-byte aligned global
// address; nothing waits for it.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    AR_GUARD_G(src, bytes, false, 16, return)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kPollSuspendNs)
        : "memory");
    return ok != 0;
}

// Plain arrival (release) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait: true when the phase with `parity` completed.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void report_error(unsigned int *err, unsigned int bits)
{
    if (err) atomicOr(err, bits);
}


// 16-byte asynchronous copy global -> shared by one thread (completes at this
// thread's next cp_async_wait_all); both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc)
{
    AR_GUARD_G(gsrc, 16, false, 16, return)
    AR_GUARD_S(smem_dst, 16, 16, return)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Named barrier `id` (1..15) over `count` threads of the block (a multiple of
// 32): bar_sync_named waits for all of them; bar_arrive_named counts this
// thread's arrival without waiting (a producer signalling waiting consumers;
// its earlier shared-memory writes are visible to them after their wait).
__device__ __forceinline__ void bar_sync_named(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive_named(int id, int count)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- 8-element chunks ------------------------------------------------------
// A chunk is 8 consecutive elements of a row: 16 bytes in bf16, 32 in fp32.

template <typename T> struct ChunkBytes;
template <> struct ChunkBytes<__nv_bfloat16> { static constexpr int value = 16; };
template <> struct ChunkBytes<float> { static constexpr int value = 32; };

__device__ __forceinline__ void unpack_bf16x8(const uint4 u, float v[8])
{
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
    v[4] = __uint_as_float(u.z << 16);
    v[5] = __uint_as_float(u.z & 0xffff0000u);
    v[6] = __uint_as_float(u.w << 16);
    v[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

// 16-byte shared-memory load issued exactly where written (volatile), so a
// second pass over a staged row re-reads shared memory instead of pinning the
// first pass's values in registers.
__device__ __forceinline__ uint4 lds128(const void *p)
{
    uint4 u;
    AR_GUARD_S(p, 16, 16, return make_uint4(0u, 0u, 0u, 0u))
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                 : "r"(smem_u32(p))
                 : "memory");
    return u;
}

// Load a chunk from shared memory (any generic pointer to smem).
__device__ __forceinline__ void ld_chunk_s(const __nv_bfloat16 *p, float v[8])
{
    unpack_bf16x8(lds128(p), v);
}
__device__ __forceinline__ void ld_chunk_s(const float *p, float v[8])
{
    const uint4 a = lds128(p);
    const uint4 b = lds128(p + 4);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}

// Load a chunk from global memory through the read-only path.
__device__ __forceinline__ void zero8(float v[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
}
__device__ __forceinline__ void ld_chunk_g(const __nv_bfloat16 *p, float v[8])
{
    AR_GUARD_G(p, 16, false, 16, return zero8(v))
    unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(p)), v);
}
__device__ __forceinline__ void ld_chunk_g(const float *p, float v[8])
{
    AR_GUARD_G(p, 32, false, 16, return zero8(v))
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Store a chunk (rounded to nearest even for bf16) through a generic pointer:
// st_chunk_g into global memory, st_chunk_s into shared memory (the same
// store; only the checked build tells them apart).
__device__ __forceinline__ void st_chunk_raw(__nv_bfloat16 *p, const float v[8])
{
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4 *>(p) = u;
}
__device__ __forceinline__ void st_chunk_raw(float *p, const float v[8])
{
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <typename T> __device__ __forceinline__ void st_chunk_g(T *p, const float v[8])
{
    AR_GUARD_G(p, (uint32_t)ChunkBytes<T>::value, true, 16, return)
    st_chunk_raw(p, v);
}
template <typename T> __device__ __forceinline__ void st_chunk_s(T *p, const float v[8])
{
    AR_GUARD_S(p, (uint32_t)ChunkBytes<T>::value, 16, return)
    st_chunk_raw(p, v);
}

// ---- packed fp32 pairs ---------------------------------------------------------
// sm_100-class GPUs execute two fp32 multiplies or FMAs as one f32x2
// instruction; each lane is rounded exactly as __fmul_rn / fmaf round, so the
// packed forms below give the bits of the scalar code they replace, with half
// the instructions. Elements e and e + 4 of a chunk share a pair (the two
// halves of the dot product below run side by side).
__device__ __forceinline__ uint64_t pk2(float x, float y)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &x, float &y)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// y[e] = fmaf(a, x[e], y[e]) for the 8 elements of a chunk.
__device__ __forceinline__ void axpy8(float a, const float x[8], float y[8])
{
    const uint64_t aa = pk2(a, a);
#pragma unroll
    for (int e = 0; e < 4; ++e) upk2(fma2(aa, pk2(x[e], x[e + 4]), pk2(y[e], y[e + 4])), y[e], y[e + 4]);
}

// Dot product of two 8-element chunks as (low half) + (high half), each half
// a fixed chain (a product, then three FMAs in element order). Exchanging the
// halves (lane-swapped order below) gives the same bits, because the final
// addition commutes exactly.
__device__ __forceinline__ float dot8(const float a[8], const float b[8])
{
    float lo = __fmul_rn(a[0], b[0]);
    lo = fmaf(a[1], b[1], lo);
    lo = fmaf(a[2], b[2], lo);
    lo = fmaf(a[3], b[3], lo);
    float hi = __fmul_rn(a[4], b[4]);
    hi = fmaf(a[5], b[5], hi);
    hi = fmaf(a[6], b[6], hi);
    hi = fmaf(a[7], b[7], hi);
    return __fadd_rn(lo, hi);
}

// dot8 with its two chains run as one packed chain: the same bits in half the
// multiply-add instructions. (Used by the forwards; in the backward kernels
// the packed forms measured slower: 1B backward 90.0 -> 91.2 ms.)
__device__ __forceinline__ float dot8p(const float a[8], const float b[8])
{
    uint64_t s = mul2(pk2(a[0], a[4]), pk2(b[0], b[4]));
#pragma unroll
    for (int e = 1; e < 4; ++e) s = fma2(pk2(a[e], a[e + 4]), pk2(b[e], b[e + 4]), s);
    float lo, hi;
    upk2(s, lo, hi);
    return __fadd_rn(lo, hi);
}

// ---- chunks in lane-swapped element order -----------------------------------
// A warp reading 32-byte fp32 chunks, one per lane, with 16-byte loads hits
// every shared-memory bank twice per quarter-warp if all lanes read the same
// half first. Lanes with sw = 4 therefore read the upper half first and keep
// their chunk's elements in swapped order: register element e holds memory
// element e ^ sw. Every per-element operand of such a lane (source values,
// dL/dout, q*g, partial sums) is kept in the same order, so the arithmetic is
// unchanged and only loads and stores see the swap.

__device__ __forceinline__ uint4 swap_halves(uint4 u, int sw)
{
    return sw ? make_uint4(u.z, u.w, u.x, u.y) : u;
}

__device__ __forceinline__ void ld_chunk_s_sw(const __nv_bfloat16 *p, int sw, float v[8])
{
    unpack_bf16x8(swap_halves(lds128(p), sw), v);
}
__device__ __forceinline__ void ld_chunk_s_sw(const float *p, int sw, float v[8])
{
    const uint4 a = lds128(p + sw);
    const uint4 b = lds128(p + (sw ^ 4));
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}
__device__ __forceinline__ void ld_chunk_g_sw(const __nv_bfloat16 *p, int sw, float v[8])
{
    AR_GUARD_G(p, 16, false, 16, return zero8(v))
    unpack_bf16x8(swap_halves(__ldg(reinterpret_cast<const uint4 *>(p)), sw), v);
}
__device__ __forceinline__ void ld_chunk_g_sw(const float *p, int sw, float v[8])
{
    AR_GUARD_G(p, 32, false, 16, return zero8(v))
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p + sw));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p + (sw ^ 4)));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st_f32x8_raw_sw(float *p, int sw, const float v[8])
{
    *reinterpret_cast<float4 *>(p + sw) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4 *>(p + (sw ^ 4)) = make_float4(v[4], v[5], v[6], v[7]);
}
// ... into global memory / into shared memory
__device__ __forceinline__ void st_f32x8_g_sw(float *p, int sw, const float v[8])
{
    AR_GUARD_G(p, 32, true, 16, return)
    st_f32x8_raw_sw(p, sw, v);
}
__device__ __forceinline__ void st_f32x8_s_sw(float *p, int sw, const float v[8])
{
    AR_GUARD_S(p, 32, 16, return)
    st_f32x8_raw_sw(p, sw, v);
}

// One fp32 chunk of a gradient row in global memory: a single 256-bit store
// (one whole 32-byte sector) when the rows' base is 32-byte aligned (v8),
// else two 16-byte stores. Lanes holding swapped halves (sw = 4) put them
// back in order.
__device__ __forceinline__ void st_grad8(float *p, int sw, const float v[8], bool v8)
{
    if (v8) {
        AR_GUARD_G(p, 32, true, 32, return)
        float x[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[e] = sw ? v[e + 4] : v[e];
            x[e + 4] = sw ? v[e] : v[e + 4];
        }
        asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                         __cvta_generic_to_global(p)),
                     "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                     "f"(x[7]));
    } else {
        st_f32x8_g_sw(p, sw, v);
    }
}

// Chunk order of a lane inside its head: rotating by the head index keeps the
// head groups that share a quarter-warp on different banks when d/256 (CPL)
// is even; for odd CPL the plain order already does.
template <int CPL>
__device__ __forceinline__ int chunk_of(int h, int sub, int LPH, int j)
{
    constexpr int rot = (CPL & 1) ? 0 : 1;
    return h * (CPL * LPH) + sub + LPH * ((j + rot * h) % CPL);
}

// fp32 chunk (gradient rows) in shared / global memory.
__device__ __forceinline__ void ld_f32x8_s(const float *p, float v[8]) { ld_chunk_s(p, v); }
__device__ __forceinline__ void st_f32x8_s(float *p, const float v[8])
{
    AR_GUARD_S(p, 32, 16, return)
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void st_f32x8_g(float *p, const float v[8]) { st_chunk_g(p, v); }

// Forward epilogue of one 8-element chunk of the routed mix o at element
// offset off: out = o, or out = partial + alpha * o in the delta form
// ("Multi-Head Attention Residuals", Appendix E, Figure 9: in the delta form
// the forward's epilogue sums the partial and the gated mix); the plain mix
// also goes to routed when
// asked for (the delta backward needs it).
template <typename T>
__device__ __forceinline__ void store_output(const RouteArgs &a, int64_t off, const float o[8])
{
    if (a.routed) st_chunk_g(static_cast<T *>(a.routed) + off, o);
    if (a.partial) {
        const float alpha = a.alpha ? __ldg(a.alpha) : 1.0f;
        float p[8], y[8];
        ld_chunk_g(static_cast<const T *>(a.partial) + off, p);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = fmaf(alpha, o[e], p[e]);
        st_chunk_g(static_cast<T *>(a.out) + off, y);
    } else {
        st_chunk_g(static_cast<T *>(a.out) + off, o);
    }
}

// One element of the storage dtype, as fp32 / rounded from fp32 (to nearest even).
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void st_elem(float *p, float v)
{
    AR_GUARD_G(p, 4, true, 4, return)
    *p = v;
}
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, float v)
{
    AR_GUARD_G(p, 2, true, 2, return)
    *p = __float2bfloat16_rn(v);
}

// Checked scalar access to global memory (a plain __ldg / store when not
// built with the checks).
__device__ __forceinline__ float ldg_chk(const float *p)
{
    AR_GUARD_G(p, 4, false, 4, return 0.f)
    return __ldg(p);
}
__device__ __forceinline__ float ld_chk(const float *p)  // plain (coherent) load
{
    AR_GUARD_G(p, 4, false, 4, return 0.f)
    return *p;
}
// Checked plain load / store of one element of any type through a generic
// pointer to global memory.
template <typename E> __device__ __forceinline__ E ld_chk_t(const E *p)
{
    AR_GUARD_G(p, (uint32_t)sizeof(E), false, (uint32_t)sizeof(E), return E{})
    return *p;
}
template <typename E> __device__ __forceinline__ void st_chk_t(E *p, E v)
{
    AR_GUARD_G(p, (uint32_t)sizeof(E), true, (uint32_t)sizeof(E), return)
    *p = v;
}
__device__ __forceinline__ uint4 ldg16_chk(const uint4 *p)
{
    AR_GUARD_G(p, 16, false, 16, return make_uint4(0u, 0u, 0u, 0u))
    return __ldg(p);
}
__device__ __forceinline__ void st16_chk(void *p, uint4 v)
{
    AR_GUARD_G(p, 16, true, 16, return)
    *reinterpret_cast<uint4 *>(p) = v;
}
__device__ __forceinline__ void st_chk(float *p, float v)
{
    AR_GUARD_G(p, 4, true, 4, return)
    *p = v;
}

// Sum over the `lph` lanes of this lane's aligned group (lph a power of two).
__device__ __forceinline__ float group_sum(float x, int lph)
{
    for (int o = 1; o < lph; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace ar

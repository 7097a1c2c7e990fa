// Host side of the C ABI declared in include/attnres.h: bank bookkeeping
// (row count, first-touch flags of the gradient rows, the record of forward
// calls that the backward must unwind in reverse), argument checks, and the
// launches. No device memory is allocated here and nothing synchronises the
// device except ar_device_error().
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "attnres.h"
#include "ar_internal.h"
#include "shapes.h"

struct ar_bank {
    int64_t T = 0;
    int d = 0, r = 0, cap = 0, inv_ld = 0;
    ar_dtype dtype = AR_BF16;
    int norm_full = 0;
    float eps = 1e-6f;
    void *rows = nullptr;
    float *inv = nullptr;
    float *grad = nullptr;
    int count = 0;
    std::vector<uint8_t> touched;     // gradient row written since zero_grad
    std::vector<int32_t> fwd_record;  // site ids of forwards not yet backpropagated
    int device = 0;
    size_t esize = 2;
};

namespace ar {

ar_status bank_device_check(const ar_bank *b)
{
    if (!b || b->device < 0) return AR_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return AR_OK;  // no usable device: the launch itself reports the failure
    }
    return dev == b->device ? AR_OK : AR_ERR_INVALID_ARG;
}

}  // namespace ar

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

ar_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return AR_OK;
    if (e == cudaErrorNotSupported) return AR_ERR_UNSUPPORTED;
    cudaGetLastError();  // clear a sticky-free launch error so the caller may retry
    return AR_ERR_CUDA;
}

ar_status on_bank_device(const ar_bank *b) { return ar::bank_device_check(b); }

// Checks shared by the forward and the backward of a site.
ar_status check_site(const ar_bank *b, const int32_t *rows, int32_t n_src, int32_t H,
                     const float *q, const float *g)
{
    if (!b || !rows || !q) return AR_ERR_INVALID_ARG;
    if (n_src < 1 || n_src > AR_MAX_SOURCES) return AR_ERR_INVALID_ARG;
    if (H < 1 || b->d % H != 0 || b->r % H != 0) return AR_ERR_SHAPE;
    int distinct = 0;
    for (int i = 0; i < n_src; ++i) {
        int k = 0;
        while (k < i && rows[k] != rows[i]) ++k;
        distinct += k == i;
    }
    if (!ar::route_supported(b->d, b->r, H, distinct, b->dtype, distinct < n_src))
        return AR_ERR_UNSUPPORTED;
    for (int i = 0; i < n_src; ++i)
        if (rows[i] < 0 || rows[i] >= b->count) return AR_ERR_INVALID_ARG;
    if (!aligned4(q) || (g && !aligned4(g))) return AR_ERR_ALIGN;
    return AR_OK;
}

// The site's distinct rows in order of first appearance, each with the number
// of times the list names it.
void distinct_rows(const int32_t *rows, int32_t n_src, std::vector<int32_t> &uniq,
                   std::vector<int32_t> &mult)
{
    uniq.clear();
    mult.clear();
    for (int i = 0; i < n_src; ++i) {
        size_t k = 0;
        while (k < uniq.size() && uniq[k] != rows[i]) ++k;
        if (k == uniq.size()) {
            uniq.push_back(rows[i]);
            mult.push_back(1);
        } else {
            ++mult[k];
        }
    }
}

void fill_common(ar::RouteArgs &a, const ar_bank *b, const int32_t *rows_in, int32_t n_in,
                 int32_t H, const float *q, const float *g, int64_t q_stride = 1,
                 int64_t g_stride = 1)
{
    std::vector<int32_t> uniq, mult;
    distinct_rows(rows_in, n_in, uniq, mult);
    const int32_t *rows = uniq.data();
    const int32_t n_src = static_cast<int32_t>(uniq.size());
    std::memset(&a, 0, sizeof(a));
    a.bank = b->rows;
    a.inv = b->inv;
    a.grad = b->grad;
    a.q = q;
    a.g = g;
    a.q_stride = q_stride;
    a.g_stride = g_stride;
    a.T = b->T;
    a.d = b->d;
    a.r = b->r;
    a.H = H;
    a.n_src = n_src;
    a.inv_ld = b->inv_ld;
    a.norm_full = b->norm_full;
    a.grad_v8 = b->grad && (reinterpret_cast<uintptr_t>(b->grad) & 31u) == 0;
    a.eps = b->eps;
    a.err = ar::device_error_word();
    for (int i = 0; i < n_src; ++i) {
        a.rows[i] = rows[i];
        if (mult[i] > 1) {
            a.has_bias = 1;
            a.bias[i] = std::log(static_cast<float>(mult[i]));
        }
    }
}


// ---- range-check table (checked build) ----------------------------------------
// The buffers one launch may touch, with the extents this library's header
// gives them; the kernels refuse any access outside them.
#ifdef AR_CHECKED
int64_t g_trim_out = 0;  // ar_checked_trim_out: bytes taken off every out span

void chk_span(ar::RouteArgs &a, const void *p, int64_t bytes, bool writable)
{
    if (!p || bytes <= 0 || a.chk.n >= ar::kCheckSpans) return;
    const uint64_t lo = reinterpret_cast<uint64_t>(p);
    a.chk.lo[a.chk.n] = lo;
    a.chk.hi[a.chk.n] = lo + static_cast<uint64_t>(bytes);
    a.chk.wr[a.chk.n] = writable ? 1 : 0;
    ++a.chk.n;
}

int64_t vec_bytes(int r, int64_t stride) { return ((int64_t)(r - 1) * stride + 1) * 4; }

// bwd: the call is a backward (lse and the outputs are read, not written)
void chk_fill(ar::RouteArgs &a, const ar_bank *b, bool bwd, size_t ws_bytes)
{
    ar::CheckTable &c = a.chk;
    std::memset(&c, 0, sizeof(c));
    const int64_t TD = b->T * (int64_t)b->d * (int64_t)b->esize;
    c.bank = reinterpret_cast<uint64_t>(b->rows);
    c.bank_row = static_cast<uint64_t>(TD);
    c.grad = reinterpret_cast<uint64_t>(b->grad);
    c.grad_row = static_cast<uint64_t>(b->T * (int64_t)b->d * 4);
    c.cap = b->cap;
    c.fault = ar::device_check_fault();
    chk_span(a, a.inv, b->T * (int64_t)b->inv_ld * 4, a.fresh1 > 0);
    chk_span(a, a.q, vec_bytes(b->r, a.q_stride), false);
    chk_span(a, a.g, vec_bytes(b->r, a.g_stride), false);
    chk_span(a, a.out, TD - g_trim_out, true);
    chk_span(a, a.lse, b->T * (int64_t)a.H * 4, !bwd);
    chk_span(a, a.fout, TD, false);
    chk_span(a, a.dout, TD, false);
    chk_span(a, a.ws, static_cast<int64_t>(ws_bytes), true);
    chk_span(a, a.partial, TD, false);
    chk_span(a, a.alpha, 4, false);
    chk_span(a, a.routed, TD, true);
    chk_span(a, a.dalpha, 4, false);
    chk_span(a, a.fresh_src, TD, false);
    chk_span(a, a.coupling, b->T * (int64_t)a.H * 4, false);
}

// the coupling pre-pass: the backward's table, the coupling buffer writable
void chk_fill_coupling(ar::RouteArgs &a, const ar_bank *b, float *coupling)
{
    chk_fill(a, b, true, 0);
    chk_span(a, coupling, b->T * (int64_t)a.H * 4, true);
}

void chk_fill_multi(ar::MultiArgs &m, const ar_bank *b)
{
    chk_fill(m.base, b, false, 0);
    const int64_t TD = b->T * (int64_t)b->d * (int64_t)b->esize;
    for (int i = 0; i < m.nq; ++i) {
        chk_span(m.base, m.q[i], vec_bytes(b->r, 1), false);
        chk_span(m.base, m.g[i], vec_bytes(b->r, 1), false);
        chk_span(m.base, m.out[i], TD - g_trim_out, true);
        chk_span(m.base, m.lse[i], b->T * (int64_t)m.base.H * 4, true);
    }
}
#define AR_CHK_FILL(a, b, bwd, ws) chk_fill((a), (b), (bwd), (ws))
#define AR_CHK_FILL_MULTI(m, b) chk_fill_multi((m), (b))
#define AR_CHK_FILL_COUPLING(a, b, c) chk_fill_coupling((a), (b), (c))

// Tables of the launches that take no RouteArgs (append, fold, token sum,
// merge, dq/dg reduction), filled in a per-thread slot: a launch copies its
// parameters when it is made.
ar::RouteArgs &chk_slot(const ar_bank *b, bool bank_rows, bool grad_rows)
{
    thread_local ar::RouteArgs a;
    std::memset(&a, 0, sizeof(a));
    ar::CheckTable &c = a.chk;
    if (bank_rows) {
        c.bank = reinterpret_cast<uint64_t>(b->rows);
        c.bank_row = static_cast<uint64_t>(b->T * (int64_t)b->d * (int64_t)b->esize);
    }
    if (grad_rows) {
        c.grad = reinterpret_cast<uint64_t>(b->grad);
        c.grad_row = static_cast<uint64_t>(b->T * (int64_t)b->d * 4);
    }
    c.cap = b->cap;
    c.fault = ar::device_check_fault();
    a.err = ar::device_error_word();
    return a;
}

// append of row new_row (its bank slot the only store target; the partial
// sum's row acc_from read), from src: a strided [T, d] view of src_bytes
// bytes, or a row of the bank itself
const ar::RouteArgs *chk_append(const ar_bank *b, int new_row, int acc_from, const void *src,
                                int64_t src_bytes)
{
    ar::RouteArgs &a = chk_slot(b, true, false);
    a.rows[0] = new_row;
    a.n_src = 1;
    a.fresh1 = 1;
    a.acc_row = acc_from;
    const uint64_t x = reinterpret_cast<uint64_t>(src), lo = a.chk.bank;
    if (a.chk.bank_row && x >= lo && x < lo + (uint64_t)b->cap * a.chk.bank_row) {
        const int row = static_cast<int>((x - lo) / a.chk.bank_row);
        if (row != new_row) a.rows[a.n_src++] = row;
    } else {
        chk_span(a, src, src_bytes, false);
    }
    chk_span(a, b->inv, b->T * (int64_t)b->inv_ld * 4, true);
    return &a;
}

const ar::RouteArgs *chk_grad_rows(const ar_bank *b, int row0, int row1, const float *out,
                                   int64_t out_bytes)
{
    ar::RouteArgs &a = chk_slot(b, false, true);
    a.rows[a.n_src++] = row0;
    if (row1 >= 0) a.rows[a.n_src++] = row1;
    chk_span(a, out, out_bytes, true);
    return &a;
}

const ar::RouteArgs *chk_merge(const ar_bank *b, int H, const void *oa, const float *la,
                               const void *ob, const float *lb, const void *out, const float *lse)
{
    ar::RouteArgs &a = chk_slot(b, false, false);
    const int64_t TD = b->T * (int64_t)b->d * (int64_t)b->esize, TH = b->T * (int64_t)H * 4;
    chk_span(a, out, TD - g_trim_out, true);
    chk_span(a, lse, TH, true);
    chk_span(a, oa, TD, false);
    chk_span(a, ob, TD, false);
    chk_span(a, la, TH, false);
    chk_span(a, lb, TH, false);
    return &a;
}

const ar::RouteArgs *chk_reduce(const ar_bank *b, const void *ws, size_t ws_bytes, const float *q,
                                int64_t qs, const float *g, int64_t gs, const float *dq,
                                const float *dg, const float *dalpha)
{
    ar::RouteArgs &a = chk_slot(b, false, false);
    chk_span(a, dq, vec_bytes(b->r, qs), true);
    chk_span(a, dg, vec_bytes(b->r, gs), true);
    chk_span(a, dalpha, 4, true);
    chk_span(a, ws, static_cast<int64_t>(ws_bytes), false);
    chk_span(a, q, vec_bytes(b->r, qs), false);
    chk_span(a, g, vec_bytes(b->r, gs), false);
    return &a;
}
#else
#define AR_CHK_FILL(a, b, bwd, ws) ((void)0)
#define AR_CHK_FILL_MULTI(m, b) ((void)0)
#define AR_CHK_FILL_COUPLING(a, b, c) ((void)0)
inline const ar::RouteArgs *chk_append(const ar_bank *, int, int, const void *, int64_t)
{
    return nullptr;
}
inline const ar::RouteArgs *chk_grad_rows(const ar_bank *, int, int, const float *, int64_t)
{
    return nullptr;
}
inline const ar::RouteArgs *chk_merge(const ar_bank *, int, const void *, const float *,
                                      const void *, const float *, const void *, const float *)
{
    return nullptr;
}
inline const ar::RouteArgs *chk_reduce(const ar_bank *, const void *, size_t, const float *,
                                       int64_t, const float *, int64_t, const float *,
                                       const float *, const float *)
{
    return nullptr;
}
#endif

}  // namespace

extern "C" {

const char *ar_status_string(ar_status s)
{
    switch (s) {
    case AR_OK: return "AR_OK";
    case AR_ERR_INVALID_ARG: return "AR_ERR_INVALID_ARG";
    case AR_ERR_SHAPE: return "AR_ERR_SHAPE";
    case AR_ERR_ALIGN: return "AR_ERR_ALIGN";
    case AR_ERR_CAPACITY: return "AR_ERR_CAPACITY";
    case AR_ERR_ORDER: return "AR_ERR_ORDER";
    case AR_ERR_CUDA: return "AR_ERR_CUDA";
    case AR_ERR_TIMEOUT: return "AR_ERR_TIMEOUT";
    case AR_ERR_UNSUPPORTED: return "AR_ERR_UNSUPPORTED";
    case AR_ERR_BOUNDS: return "AR_ERR_BOUNDS";
    }
    return "AR_ERR_UNKNOWN";
}

ar_status ar_inv_rms_floats(int64_t T, int32_t capacity, int64_t *floats)
{
    if (!floats || T < 0 || capacity < 1) return AR_ERR_INVALID_ARG;
    *floats = T * (int64_t)((capacity + 3) / 4 * 4);
    return AR_OK;
}

ar_status ar_bank_create(ar_bank **out, int64_t T, int32_t d, int32_t r, int32_t capacity,
                         ar_dtype dtype, ar_norm norm, float eps, void *rows, float *inv_rms,
                         float *grad)
{
    if (!out) return AR_ERR_INVALID_ARG;
    *out = nullptr;
    if (capacity < 1 || T < 0) return AR_ERR_INVALID_ARG;
    if (T > 0 && (!rows || !inv_rms)) return AR_ERR_INVALID_ARG;
    if (dtype != AR_F32 && dtype != AR_BF16) return AR_ERR_INVALID_ARG;
    if (norm != AR_NORM_KEY && norm != AR_NORM_FULL) return AR_ERR_INVALID_ARG;
    if (d < 1 || r < 1 || r > d) return AR_ERR_SHAPE;
    if (!aligned16(rows) || !aligned16(inv_rms) || (grad && !aligned16(grad))) return AR_ERR_ALIGN;
    int dev = -1;  // launches use the current device; every call checks it is this one
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        dev = -1;
    }
    ar_bank *b = new (std::nothrow) ar_bank();
    if (!b) return AR_ERR_INVALID_ARG;
    b->T = T;
    b->d = d;
    b->r = r;
    b->cap = capacity;
    b->inv_ld = (capacity + 3) / 4 * 4;
    b->dtype = dtype;
    b->norm_full = norm == AR_NORM_FULL ? 1 : 0;
    b->eps = eps;
    b->rows = rows;
    b->inv = inv_rms;
    b->grad = grad;
    b->touched.assign(static_cast<size_t>(capacity), 0);
    b->device = dev;
    b->esize = dtype == AR_BF16 ? 2 : 4;
    *out = b;
    return AR_OK;
}

ar_status ar_bank_destroy(ar_bank *bank)
{
    delete bank;
    return AR_OK;
}

ar_status ar_bank_row_count(const ar_bank *bank, int32_t *count)
{
    if (!bank || !count) return AR_ERR_INVALID_ARG;
    *count = bank->count;
    return AR_OK;
}

ar_status ar_bank_row_ptr(const ar_bank *bank, int32_t row, void **ptr)
{
    if (!bank || !ptr || row < 0 || row >= bank->cap) return AR_ERR_INVALID_ARG;
    *ptr = static_cast<unsigned char *>(bank->rows) +
           (size_t)row * (size_t)bank->T * (size_t)bank->d * bank->esize;
    return AR_OK;
}

ar_status ar_bank_append_strided(ar_bank *bank, const void *src, int64_t token_stride,
                                 int64_t elem_stride, int32_t accumulate_from, int32_t *out_row,
                                 void *stream)
{
    if (!bank || (!src && bank->T > 0)) return AR_ERR_INVALID_ARG;
    if (token_stride < 0 || elem_stride < 1) return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (bank->count >= bank->cap) return AR_ERR_CAPACITY;
    if (accumulate_from < -1 || accumulate_from >= bank->count) return AR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) % bank->esize) != 0) return AR_ERR_ALIGN;
    void *dst = nullptr;
    ar_bank_row_ptr(bank, bank->count, &dst);
    const void *prev = nullptr;
    if (accumulate_from >= 0) ar_bank_row_ptr(bank, accumulate_from, const_cast<void **>(&prev));
    const int64_t src_bytes =
        bank->T > 0 ? ((bank->T - 1) * token_stride + (int64_t)(bank->d - 1) * elem_stride + 1) *
                          (int64_t)bank->esize
                    : 0;
    const cudaError_t e = ar::launch_append(
        src, prev, dst, bank->inv + bank->count, bank->T, bank->d, bank->r, bank->inv_ld,
        bank->norm_full, bank->eps, bank->dtype, static_cast<cudaStream_t>(stream), token_stride,
        elem_stride, chk_append(bank, bank->count, accumulate_from, src, src_bytes));
    if (e != cudaSuccess) return from_cuda(e);
    if (out_row) *out_row = bank->count;
    ++bank->count;
    return AR_OK;
}

ar_status ar_bank_append(ar_bank *bank, const void *src, int32_t accumulate_from,
                         int32_t *out_row, void *stream)
{
    return ar_bank_append_strided(bank, src, bank ? bank->d : 0, 1, accumulate_from, out_row,
                                  stream);
}

ar_status ar_bank_zero_grad(ar_bank *bank)
{
    if (!bank) return AR_ERR_INVALID_ARG;
    std::fill(bank->touched.begin(), bank->touched.end(), 0);
    return AR_OK;
}

ar_status ar_bank_reset(ar_bank *bank)
{
    if (!bank) return AR_ERR_INVALID_ARG;
    bank->count = 0;
    bank->fwd_record.clear();
    std::fill(bank->touched.begin(), bank->touched.end(), 0);
    return AR_OK;
}

namespace {

ar_status route_fwd_impl(ar_bank *bank, const ar_site &st_, const void *partial,
                         const float *alpha, void *out, void *routed, float *lse, void *stream)
{
    const int32_t *rows = st_.rows;
    const int32_t n_src = st_.n_src, H = st_.H;
    const float *q = st_.q, *g = st_.g;
    if (st_.q_stride < 1 || (g && st_.g_stride < 1)) return AR_ERR_INVALID_ARG;
    ar_status st = check_site(bank, rows, n_src, H, q, g);
    if (st != AR_OK) return st;
    if (bank->T > 0 && (!out || !lse)) return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned4(lse) || !aligned16(partial) || !aligned16(routed) ||
        !aligned4(alpha))
        return AR_ERR_ALIGN;
    if ((partial || alpha || routed) && !(partial && alpha && routed)) return AR_ERR_INVALID_ARG;
    if (bank->T > 0) {
        ar::RouteArgs a;
        fill_common(a, bank, rows, n_src, H, q, g, st_.q_stride, st_.g_stride);
        a.out = out;
        a.lse = lse;
        a.partial = partial;
        a.alpha = alpha;
        a.routed = routed;
        AR_CHK_FILL(a, bank, false, 0);
        const cudaError_t e = ar::launch_route_fwd(a, bank->dtype, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return from_cuda(e);
    }
    bank->fwd_record.push_back(st_.site_id);
    return AR_OK;
}

ar_site make_site(const int32_t *rows, int32_t n_src, int32_t H, const float *q, const float *g,
                  int32_t site_id)
{
    ar_site s;
    s.rows = rows;
    s.n_src = n_src;
    s.H = H;
    s.q = q;
    s.q_stride = 1;
    s.g = g;
    s.g_stride = 1;
    s.site_id = site_id;
    return s;
}

}  // namespace

ar_status ar_route_fwd(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                       const float *q, const float *g, void *out, float *lse, int32_t site_id,
                       void *stream)
{
    return route_fwd_impl(bank, make_site(rows, n_src, H, q, g, site_id), nullptr, nullptr, out,
                          nullptr, lse, stream);
}

ar_status ar_route_fwd_append(ar_bank *bank, const void *src, int32_t accumulate_from,
                              int32_t *out_row, const int32_t *rows, int32_t n_src, int32_t H,
                              const float *q, const float *g, void *out, float *lse,
                              int32_t site_id, int32_t *fused, void *stream)
{
    if (fused) *fused = 0;
    if (!bank || (!src && bank->T > 0)) return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (bank->count >= bank->cap) return AR_ERR_CAPACITY;
    if (accumulate_from < -1 || accumulate_from >= bank->count) return AR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) % bank->esize) != 0) return AR_ERR_ALIGN;
    // the site's checks, with the new row counted, before anything happens
    const int32_t new_row = bank->count;
    ++bank->count;
    ar_status st = check_site(bank, rows, n_src, H, q, g);
    if (st == AR_OK && bank->T > 0 && (!out || !lse)) st = AR_ERR_INVALID_ARG;
    if (st == AR_OK && (!aligned16(out) || !aligned4(lse))) st = AR_ERR_ALIGN;
    --bank->count;
    if (st != AR_OK) return st;

    void *slot = nullptr;
    ar_bank_row_ptr(bank, new_row, &slot);
    const bool in_place = src == slot && accumulate_from < 0;
    if (bank->T > 0 && (in_place || aligned16(src))) {
        // the forward forms the row (copy or partial sum) where needed and
        // computes its inverse RMS
        ++bank->count;
        ar::RouteArgs a;
        fill_common(a, bank, rows, n_src, H, q, g);
        int idx = -1;
        for (int i = 0; i < a.n_src; ++i)
            if (a.rows[i] == new_row) idx = i;
        if (idx >= 0 && ar::fwd_fuses_append(a, bank->dtype, in_place)) {
            a.fresh1 = idx + 1;
            a.fresh_src = in_place ? nullptr : src;
            a.acc_row = accumulate_from;
            a.out = out;
            a.lse = lse;
            AR_CHK_FILL(a, bank, false, 0);
            const cudaError_t e =
                ar::launch_route_fwd(a, bank->dtype, static_cast<cudaStream_t>(stream));
            if (e != cudaSuccess) {
                --bank->count;
                return from_cuda(e);
            }
            bank->fwd_record.push_back(site_id);
            if (out_row) *out_row = new_row;
            if (fused) *fused = 1;
            return AR_OK;
        }
        --bank->count;
    }
    st = ar_bank_append(bank, src, accumulate_from, out_row, stream);
    if (st != AR_OK) return st;
    return ar_route_fwd(bank, rows, n_src, H, q, g, out, lse, site_id, stream);
}

ar_status ar_route_fwd_delta(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                             const float *q, const float *g, const void *partial,
                             const float *alpha, void *out, void *routed, float *lse,
                             int32_t site_id, void *stream)
{
    if (bank && bank->T > 0 && (!partial || !alpha || !routed)) return AR_ERR_INVALID_ARG;
    return route_fwd_impl(bank, make_site(rows, n_src, H, q, g, site_id), partial, alpha, out,
                          routed, lse, stream);
}

ar_status ar_route_fwd_site(ar_bank *bank, const ar_site *site, const void *partial,
                            const float *alpha, void *out, void *routed, float *lse, void *stream)
{
    if (!site) return AR_ERR_INVALID_ARG;
    return route_fwd_impl(bank, *site, partial, alpha, out, routed, lse, stream);
}

ar_status ar_route_fwd_multi(const ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                             int32_t n_q, const float *const *q, const float *const *g,
                             void *const *out, float *const *lse, void *stream)
{
    if (!bank || !rows || !q) return AR_ERR_INVALID_ARG;
    if (n_src < 1 || n_src > AR_MAX_SOURCES) return AR_ERR_INVALID_ARG;
    if (n_q < 1 || n_q > AR_MAX_QUERIES) return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (H < 1 || bank->d % H != 0 || bank->r % H != 0) return AR_ERR_SHAPE;
    for (int i = 0; i < n_src; ++i)
        if (rows[i] < 0 || rows[i] >= bank->count) return AR_ERR_INVALID_ARG;
    for (int i = 0; i < n_q; ++i) {
        if (!q[i]) return AR_ERR_INVALID_ARG;
        if (!aligned4(q[i]) || (g && g[i] && !aligned4(g[i]))) return AR_ERR_ALIGN;
        if (bank->T > 0) {
            if (!out || !lse || !out[i] || !lse[i]) return AR_ERR_INVALID_ARG;
            if (!aligned16(out[i]) || !aligned4(lse[i])) return AR_ERR_ALIGN;
        }
    }
    if (bank->T == 0) return AR_OK;
    ar::MultiArgs m;
    std::memset(&m, 0, sizeof(m));
    fill_common(m.base, bank, rows, n_src, H, q[0], g ? g[0] : nullptr);
    m.nq = n_q;
    for (int i = 0; i < n_q; ++i) {
        m.q[i] = q[i];
        m.g[i] = g ? g[i] : nullptr;
        m.out[i] = out[i];
        m.lse[i] = lse[i];
    }
    AR_CHK_FILL_MULTI(m, bank);
    const cudaError_t e = ar::launch_route_fwd_multi(m, bank->dtype, static_cast<cudaStream_t>(stream));
    return from_cuda(e);
}

ar_status ar_route_bwd_workspace(const ar_bank *bank, int32_t H, size_t *bytes)
{
    if (!bank || !bytes) return AR_ERR_INVALID_ARG;
    if (H < 1 || bank->d % H != 0 || bank->r % H != 0) return AR_ERR_SHAPE;
    if (!ar::route_supported(bank->d, bank->r, H, 1, bank->dtype, false)) return AR_ERR_UNSUPPORTED;
    ar::RouteArgs a;
    std::memset(&a, 0, sizeof(a));
    a.d = bank->d;
    a.r = bank->r;
    a.H = H;
    a.n_src = 1;
    int warps = 0;
    cudaError_t e = ar::route_bwd_grid(a, bank->dtype, &warps);
    if (e != cudaSuccess) return from_cuda(e);
    // the exact-coupling variant of the kernels (ar_route_bwd_exact) may
    // keep more blocks resident: the workspace serves both
    static const float kAnyCoupling = 0.f;
    a.coupling = &kAnyCoupling;
    int warps_cs = 0;
    e = ar::route_bwd_grid(a, bank->dtype, &warps_cs);
    if (e != cudaSuccess) return from_cuda(e);
    warps = std::max(warps, warps_cs);
    // any site may run on the scalar-access kernels (repeated rows, or more
    // sources than the sliced-key kernels' key cache holds)
    int gw = 0;
    e = ar::generic_bwd_rows(&gw);
    if (e != cudaSuccess) return from_cuda(e);
    warps = std::max(warps, gw);
    // [rows, r] partial sums of dq/dg, then a [rows, 4] tail for dL/dalpha
    *bytes = (size_t)warps * ((size_t)bank->r + 4) * sizeof(float);
    return AR_OK;
}

namespace {

ar_status route_bwd_impl(ar_bank *bank, const ar_site &st_, const void *out, const void *dout,
                         const float *lse, const float *alpha, float *dq, float *dg,
                         float *dalpha, void *ws, size_t ws_bytes, void *stream,
                         float *coupling = nullptr)
{
    const int32_t *rows = st_.rows;
    const int32_t n_src = st_.n_src, H = st_.H;
    const float *q = st_.q, *g = st_.g;
    if (st_.q_stride < 1 || (g && st_.g_stride < 1)) return AR_ERR_INVALID_ARG;
    if (bank && !bank->grad && bank->T > 0) return AR_ERR_INVALID_ARG;
    ar_status st = check_site(bank, rows, n_src, H, q, g);
    if (st != AR_OK) return st;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (!dq || (bank->T > 0 && (!out || !dout || !lse || !ws))) return AR_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(dout) || !aligned4(lse) || !aligned4(dq) ||
        (dg && !aligned4(dg)) || !aligned16(ws) || !aligned4(alpha) || !aligned4(dalpha))
        return AR_ERR_ALIGN;
    if ((alpha != nullptr) != (dalpha != nullptr)) return AR_ERR_INVALID_ARG;
    if (bank->fwd_record.empty() || bank->fwd_record.back() != st_.site_id) return AR_ERR_ORDER;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (bank->T == 0) {
        // no tokens: the reduction over zero workspace rows writes zeros
        const cudaError_t e = ar::launch_dqdg_reduce(
            static_cast<const float *>(ws), 0, bank->r, q, st_.q_stride, g, st_.g_stride, dq, dg,
            dalpha, s,
            chk_reduce(bank, ws, ws_bytes, q, st_.q_stride, g, st_.g_stride, dq, dg, dalpha));
        if (e != cudaSuccess) return from_cuda(e);
    } else {
        ar::RouteArgs a;
        fill_common(a, bank, rows, n_src, H, q, g, st_.q_stride, st_.g_stride);
        a.fout = out;
        a.dout = dout;
        a.lse = const_cast<float *>(lse);
        a.ws = static_cast<float *>(ws);
        a.alpha = alpha;
        a.dalpha = dalpha;
        for (int i = 0; i < a.n_src; ++i)
            if (!bank->touched[a.rows[i]]) a.first_mask[i >> 5] |= 1u << (i & 31);
        // the kernel variant (and so its grid) depends on where the coupling
        // term comes from
        a.coupling = coupling;
        // workspace rows of the family serving this site (at most what
        // ar_route_bwd_workspace reports)
        int ws_rows = 0;
        cudaError_t e = ar::route_bwd_grid(a, bank->dtype, &ws_rows);
        if (e != cudaSuccess) return from_cuda(e);
        if (ws_bytes < (size_t)ws_rows * ((size_t)bank->r + 4) * sizeof(float))
            return AR_ERR_CAPACITY;
        if (coupling) {
            // the coupling term summed over the sources first, then read by
            // the backward in place of <G_h, out_h>
            AR_CHK_FILL_COUPLING(a, bank, coupling);
            e = ar::launch_route_coupling(a, coupling, bank->dtype, s);
            if (e != cudaSuccess) return from_cuda(e);
        }
        AR_CHK_FILL(a, bank, true, ws_bytes);
        e = ar::launch_route_bwd(a, bank->dtype, s);
        if (e != cudaSuccess) return from_cuda(e);
        e = ar::launch_dqdg_reduce(
            static_cast<const float *>(ws), ws_rows, bank->r, q, st_.q_stride, g, st_.g_stride, dq,
            dg, dalpha, s,
            chk_reduce(bank, ws, ws_bytes, q, st_.q_stride, g, st_.g_stride, dq, dg, dalpha));
        if (e != cudaSuccess) return from_cuda(e);
    }
    for (int i = 0; i < n_src; ++i) bank->touched[rows[i]] = 1;
    bank->fwd_record.pop_back();
    return AR_OK;
}

}  // namespace

ar_status ar_route_bwd(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                       const float *q, const float *g, const void *out, const void *dout,
                       const float *lse, float *dq, float *dg, void *ws, size_t ws_bytes,
                       int32_t site_id, void *stream)
{
    return route_bwd_impl(bank, make_site(rows, n_src, H, q, g, site_id), out, dout, lse, nullptr,
                          dq, dg, nullptr, ws, ws_bytes, stream);
}

ar_status ar_route_bwd_delta(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                             const float *q, const float *g, const void *routed, const void *dout,
                             const float *lse, const float *alpha, float *dq, float *dg,
                             float *dalpha, void *ws, size_t ws_bytes, int32_t site_id,
                             void *stream)
{
    if (!alpha || !dalpha) return AR_ERR_INVALID_ARG;
    return route_bwd_impl(bank, make_site(rows, n_src, H, q, g, site_id), routed, dout, lse, alpha,
                          dq, dg, dalpha, ws, ws_bytes, stream);
}

ar_status ar_route_bwd_site(ar_bank *bank, const ar_site *site, const void *out, const void *dout,
                            const float *lse, const float *alpha, float *dq, float *dg,
                            float *dalpha, void *ws, size_t ws_bytes, void *stream)
{
    if (!site) return AR_ERR_INVALID_ARG;
    return route_bwd_impl(bank, *site, out, dout, lse, alpha, dq, dg, dalpha, ws, ws_bytes, stream);
}

ar_status ar_route_bwd_exact(ar_bank *bank, const ar_site *site, const void *out,
                             const void *dout, const float *lse, const float *alpha,
                             float *coupling, float *dq, float *dg, float *dalpha, void *ws,
                             size_t ws_bytes, void *stream)
{
    if (!site) return AR_ERR_INVALID_ARG;
    if (alpha || dalpha) return AR_ERR_UNSUPPORTED;   // the plain form only
    if (bank && bank->T > 0 && !coupling) return AR_ERR_INVALID_ARG;
    if (!aligned4(coupling)) return AR_ERR_ALIGN;
    return route_bwd_impl(bank, *site, out, dout, lse, alpha, dq, dg, dalpha, ws, ws_bytes, stream,
                          coupling);
}

ar_status ar_bank_append_broadcast(ar_bank *bank, const void *vec, int32_t *out_row, void *stream)
{
    if (!bank || !vec) return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (bank->count >= bank->cap) return AR_ERR_CAPACITY;
    if ((reinterpret_cast<uintptr_t>(vec) % bank->esize) != 0) return AR_ERR_ALIGN;
    void *dst = nullptr;
    ar_bank_row_ptr(bank, bank->count, &dst);
    const cudaError_t e = ar::launch_append(
        vec, nullptr, dst, bank->inv + bank->count, bank->T, bank->d, bank->r, bank->inv_ld,
        bank->norm_full, bank->eps, bank->dtype, static_cast<cudaStream_t>(stream), 0, 1,
        chk_append(bank, bank->count, -1, vec, (int64_t)bank->d * (int64_t)bank->esize));
    if (e != cudaSuccess) return from_cuda(e);
    if (out_row) *out_row = bank->count;
    ++bank->count;
    return AR_OK;
}

ar_status ar_bank_grad_token_sum(const ar_bank *bank, int32_t row, float *out, void *stream)
{
    if (!bank || !out || row < 0 || row >= bank->count) return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (!bank->grad && bank->T > 0) return AR_ERR_INVALID_ARG;
    if (!aligned4(out)) return AR_ERR_ALIGN;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (bank->T == 0 || !bank->touched[row])
        e = cudaMemsetAsync(out, 0, (size_t)bank->d * sizeof(float), s);
    else
        e = ar::launch_token_sum(bank->grad + (int64_t)row * bank->T * bank->d, bank->T, bank->d,
                                 out, s, chk_grad_rows(bank, row, -1, out, (int64_t)bank->d * 4));
    return e == cudaSuccess ? AR_OK : from_cuda(e);
}

ar_status ar_bank_grad_fold(ar_bank *bank, int32_t dst_row, int32_t src_row, void *stream)
{
    if (!bank || dst_row < 0 || src_row < 0 || dst_row >= bank->count ||
        src_row >= bank->count || dst_row == src_row)
        return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (!bank->grad) return bank->T == 0 ? AR_OK : AR_ERR_INVALID_ARG;
    const int64_t n = bank->T * (int64_t)bank->d;
    float *dst = bank->grad + (int64_t)dst_row * n;
    const float *src = bank->grad + (int64_t)src_row * n;
    const cudaError_t e = ar::launch_grad_fold(dst, src, n, bank->touched[src_row] != 0,
                                               bank->touched[dst_row] != 0,
                                               static_cast<cudaStream_t>(stream),
                                               chk_grad_rows(bank, dst_row, src_row, nullptr, 0));
    if (e != cudaSuccess) return from_cuda(e);
    bank->touched[dst_row] = 1;
    return AR_OK;
}

ar_status ar_route_merge(const ar_bank *bank, int32_t H, const void *out_a, const float *lse_a,
                         const void *out_b, const float *lse_b, void *out, float *lse, void *stream)
{
    if (!bank) return AR_ERR_INVALID_ARG;
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    if (H < 1 || bank->d % H != 0) return AR_ERR_SHAPE;
    if (bank->T > 0 && (!out_a || !lse_a || !out_b || !lse_b || !out || !lse))
        return AR_ERR_INVALID_ARG;
    if (!aligned16(out_a) || !aligned16(out_b) || !aligned16(out) || !aligned4(lse_a) ||
        !aligned4(lse_b) || !aligned4(lse))
        return AR_ERR_ALIGN;
    const cudaError_t e = ar::launch_merge(out_a, lse_a, out_b, lse_b, out, lse, bank->T, bank->d,
                                           H, bank->dtype, static_cast<cudaStream_t>(stream),
                                           chk_merge(bank, H, out_a, lse_a, out_b, lse_b, out, lse));
    return e == cudaSuccess ? AR_OK : from_cuda(e);
}

ar_status ar_block_schedule(int32_t M, int32_t NB, int32_t *acc_from, int32_t *site_ptr,
                            int32_t *site_rows, int64_t site_rows_cap, int64_t *site_rows_len)
{
    if (M < 1 || !acc_from || !site_ptr || !site_rows_len) return AR_ERR_INVALID_ARG;
    const int64_t nb = (NB <= 0 || NB >= M) ? M : NB;
    std::vector<uint8_t> is_end(static_cast<size_t>(M) + 1, 0);
    for (int64_t j = 1; j <= nb; ++j) is_end[(M * j + nb - 1) / nb] = 1;  // ceil(M j / NB)
    // Row t holds its block's running sum up to sublayer t: a copy of o_t when
    // t opens a block (t = 1, or t - 1 closed one), else row t - 1 plus o_t.
    // The read after sublayer t lists row 0, the last row of every block
    // closed before t, and row t.
    std::vector<int32_t> closed;  // last rows of the blocks closed so far
    std::vector<int32_t> flat{0};
    std::vector<int32_t> ptr{0, 1};
    acc_from[0] = -1;
    for (int32_t t = 1; t <= M; ++t) {
        const bool opens = t == 1 || is_end[t - 1];
        acc_from[t] = opens ? -1 : t - 1;
        flat.push_back(0);
        flat.insert(flat.end(), closed.begin(), closed.end());
        flat.push_back(t);
        ptr.push_back(static_cast<int32_t>(flat.size()));
        if (is_end[t]) closed.push_back(t);
    }
    *site_rows_len = static_cast<int64_t>(flat.size());
    for (int32_t t = 0; t <= M + 1; ++t) site_ptr[t] = ptr[t];
    if (!site_rows || site_rows_cap < (int64_t)flat.size()) return AR_ERR_CAPACITY;
    std::memcpy(site_rows, flat.data(), flat.size() * sizeof(int32_t));
    return AR_OK;
}

ar_status ar_route_fwd_lost_copies(ar_bank *bank, const int32_t *rows, int32_t n_src,
                                   int32_t H, const float *q, const float *g, void *out,
                                   float *lse, uint32_t poll_limit, void *stream)
{
    if (on_bank_device(bank) != AR_OK) return AR_ERR_INVALID_ARG;
    ar_status st = check_site(bank, rows, n_src, H, q, g);
    if (st != AR_OK) return st;
    if (poll_limit < 1 || bank->T < 1 || !out || !lse) return AR_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned4(lse)) return AR_ERR_ALIGN;
    // the one-warp full-key forward: full keys, rows of 768 to 2048 columns
    // (narrower rows with at most 4 heads take the two-tokens-per-warp kernel)
    const size_t es = bank->dtype == AR_BF16 ? 2 : 4;
    if (ar::family_of(bank->d, bank->r, H, n_src, es, false) != ar::Family::kFull ||
        (bank->d <= 512 && H <= 4))
        return AR_ERR_UNSUPPORTED;
    ar::RouteArgs a;
    fill_common(a, bank, rows, n_src, H, q, g);
    if (a.has_bias) return AR_ERR_UNSUPPORTED;
    a.out = out;
    a.lse = lse;
    a.wait_limit = poll_limit;
    a.lost_copies = 1;
    AR_CHK_FILL(a, bank, false, 0);
    return from_cuda(ar::launch_route_fwd(a, bank->dtype, static_cast<cudaStream_t>(stream)));
}

ar_status ar_device_status(void)
{
    uint32_t bits = 0;
    const ar_status st = ar_device_error(&bits);
    if (st != AR_OK) return st;
    if (bits & AR_DEVERR_BOUNDS) return AR_ERR_BOUNDS;
    return (bits & AR_DEVERR_WAIT_TIMEOUT) ? AR_ERR_TIMEOUT : AR_OK;
}

ar_status ar_checked_fault(int32_t *checked, uint64_t *addr, uint32_t *bytes, uint32_t *kind)
{
    if (!checked || !addr || !bytes || !kind) return AR_ERR_INVALID_ARG;
    *checked = 0;
    *addr = 0;
    *bytes = 0;
    *kind = 0;
#ifdef AR_CHECKED
    *checked = 1;
    unsigned long long *f = ar::device_check_fault();
    unsigned long long v[3] = {0ull, 0ull, 0ull};
    if (!f || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(v, f, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(f, 0, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_CUDA;
    }
    if (v[0]) {
        *addr = v[1];
        *bytes = static_cast<uint32_t>(v[2] & 0xffffffffull);
        *kind = static_cast<uint32_t>(v[2] >> 32);
    }
#endif
    return AR_OK;
}

ar_status ar_checked_trim_out(int64_t bytes)
{
#ifdef AR_CHECKED
    if (bytes < 0) return AR_ERR_INVALID_ARG;
    g_trim_out = bytes;
    return AR_OK;
#else
    (void)bytes;
    return AR_ERR_UNSUPPORTED;
#endif
}

ar_status ar_device_error(uint32_t *bits)
{
    if (!bits) return AR_ERR_INVALID_ARG;
    unsigned int *w = ar::device_error_word();
    if (!w) {
        cudaGetLastError();
        return AR_ERR_CUDA;
    }
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(w, 0, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_CUDA;
    }
    *bits = v;
    return AR_OK;
}

}  // extern "C"

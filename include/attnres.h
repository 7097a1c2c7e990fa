/*
 * attnres.h — C ABI of the GB300 depth-routing library (libattnres_gb300.so).
 *
 * The depth-routing read of attention residuals: at every routing site each
 * token reads a learned softmax mixture over a bank of earlier sublayer
 * outputs ("Multi-Head Attention Residuals", Sec. 2.2 Eq. 2 and Sec. 2.3
 * Eq. 3; "Low-Rank Attention Residuals", Sec. 3.1-3.3 Eq. 2-12).
 *
 *   key of source n, token t : RMSNorm over the key coordinates, times g.
 *                              The key coordinates are the last r of the d
 *                              coordinates (r = d: plain AttnRes / MHAR keys;
 *                              r < d: the sliced keys of LR-AttnRes, Eq. 11).
 *   head h (H heads)         : value slice = coordinates [h*d/H, (h+1)*d/H),
 *                              key slice   = coordinates d-r + [h*r/H, (h+1)*r/H).
 *   score    z[n,h]  = inv[n] * sum_{c in key slice h} q[c'] g[c'] s_n[c]
 *                      (c' = c - (d - r): q and g are indexed over the key
 *                      coordinates), inv[n] = (mean_{key coords} s_n^2 + eps)^(-1/2)
 *   weights  a[n,h]  = softmax over n of z[.,h]            (per head; Eq. 3)
 *   output   out[c]  = sum_n a[n,h(c)] s_n[c]                          (Eq. 3)
 *   lse[h]           = log sum_n exp z[n,h]          (saved for the backward)
 * H = 1 is single-head AttnRes (MHAR Appendix B, Figure 7); r = d with H > 1 is
 * MHAR; r < d is LR-AttnRes with the heads laid over the key slice.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Memory: the caller owns all device memory and every stream. The library
 *   never allocates device memory and never synchronises the device, except
 *   in ar_device_error(), which says so. Compute calls are asynchronous on
 *   the given stream (a cudaStream_t passed as void*; NULL = legacy default).
 * - Pointers named "device" must be device-accessible; "host" pointers are
 *   read before the call returns and may be reused at once.
 * - Every call returns an ar_status. Argument checks happen on the host
 *   before anything is launched; a failed check launches nothing and leaves
 *   the bank unchanged. A CUDA launch error returns AR_ERR_CUDA.
 * - A device-side wait that runs out (a copy that never lands) does not trap:
 *   the kernel records it in a device error word and returns; read it with
 *   ar_device_error().
 * - Banks are not thread-safe; distinct banks may be used from distinct
 *   threads.
 * - A bank belongs to the device that was current when it was created.
 *   Every call that launches work on a bank's buffers runs on the current
 *   device and returns AR_ERR_INVALID_ARG, launching nothing, when that is
 *   not the bank's device.
 *
 * Shapes: every d >= 1, 1 <= r <= d and H dividing both d and r are served.
 * The tiled kernels (bulk copies into shared memory, 16-byte accesses) take
 * d a multiple of 256 with r a multiple of 8 and:
 *   - r = d <= 2048, H in {1,2,4,8,16,32};
 *   - d a multiple of 1024 up to 8192, H a multiple of 4 with H/4 in
 *     {1,2,4,8,16,32}, and r = d or r = k*d/4 (k = 1, 2) with H/k a power of
 *     two <= 32;
 *   - other r <= d with d <= 4096, H in {1,...,32} a power of two, r/H a
 *     multiple of 8 and r <= 4096 (the forward's key cache,
 *     2*n_src*r*sizeof(dtype) bytes, within 200 KB).
 * Every other shape, and every site that lists a row twice, runs on the
 * scalar-access kernels ("Low-Rank Attention Residuals", Appendix I:
 * unaligned widths such as d = 513, repeated sources), which hold the
 * site's [n_src, H] scores per warp in shared memory and return
 * AR_ERR_UNSUPPORTED only when even one warp's arrays exceed 200 KB
 * (about n_src*H > 20000). Row/output pointers must be 16-byte aligned
 * (AR_ERR_ALIGN otherwise); the delta form is served by every family except
 * the one-warp sliced-key kernels of the third item.
 */
#ifndef ATTNRES_H
#define ATTNRES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AR_MAX_SOURCES 256
#define AR_MAX_QUERIES 8

typedef enum {
    AR_OK = 0,
    AR_ERR_INVALID_ARG = 1, /* null or out-of-range argument               */
    AR_ERR_SHAPE = 2,       /* inconsistent sizes (d % H, r > d, ...)       */
    AR_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned      */
    AR_ERR_CAPACITY = 4,    /* bank full, or workspace too small            */
    AR_ERR_ORDER = 5,       /* backward not in reverse forward order        */
    AR_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed         */
    AR_ERR_TIMEOUT = 7,     /* a device-side wait ran out (see ar_device_error) */
    AR_ERR_UNSUPPORTED = 8, /* valid, but outside the fused kernels' shapes */
    AR_ERR_BOUNDS = 9       /* checked build: an access left its buffers     */
} ar_status;

typedef enum { AR_F32 = 0, AR_BF16 = 1 } ar_dtype;

/* Which coordinates the RMS statistic of a key runs over.
 * AR_NORM_KEY : the key coordinates (last r) — LR-AttnRes Eq. 13, first line;
 *               with r = d this is the full-width RMS of MHAR Appendix E.
 * AR_NORM_FULL: all d coordinates with the sliced numerator — the
 *               full-width-RMS control of LR-AttnRes Eq. 13, second line. */
typedef enum { AR_NORM_KEY = 0, AR_NORM_FULL = 1 } ar_norm;

/* Device error bits reported by ar_device_error(). */
#define AR_DEVERR_WAIT_TIMEOUT 1u
/* Set only by a library built with the range checks (see ar_checked_fault). */
#define AR_DEVERR_BOUNDS 2u

typedef struct ar_bank ar_bank; /* opaque host-side handle */

/* Human-readable name of a status. Never NULL. */
const char *ar_status_string(ar_status s);

/* Number of floats the inverse-RMS cache of a bank needs: T * ld, where
 * ld = capacity rounded up to a multiple of 4 (token-major layout, below). */
ar_status ar_inv_rms_floats(int64_t T, int32_t capacity, int64_t *floats);

/*
 * Create a bank: the single source store of MHAR Appendix E (every source row
 * lives in one preallocated tensor with a slot per sublayer output plus the
 * embedding, each slot filled once), the per-row inverse-RMS cache, and the
 * fp32 gradient rows that every site's backward adds into (Appendix E,
 * backward).
 *   T        : tokens (batch x sequence), T >= 0. T = 0 makes every compute
 *              call a no-op (the backward still zeroes dq/dg), and then every
 *              per-token pointer (rows, inv_rms, src, out, lse, dout, ws) may
 *              be NULL.
 *   d, r     : width and key width (1 <= r <= d)
 *   capacity : rows the bank can hold (1 <= capacity)
 *   dtype    : storage type of rows, outputs and dout
 *   norm     : RMS coordinates of the keys (ar_norm)
 *   eps      : RMSNorm epsilon (> 0 recommended; 1e-6 in the pages' models)
 *   rows     : device [capacity, T, d] of dtype (row-major: row j's token t
 *              starts at (j*T + t)*d elements)
 *   inv_rms  : device float [T, ld] (token-major; ld from ar_inv_rms_floats)
 *   grad     : device float [capacity, T, d], or NULL for forward-only use
 * On success *out receives a handle owned by the caller (ar_bank_destroy).
 * The pointed-to buffers must outlive the bank. Errors: AR_ERR_INVALID_ARG
 * (null out/rows/inv_rms, capacity < 1), AR_ERR_SHAPE (r > d, d < 1),
 * AR_ERR_ALIGN. Creating a bank touches no device; the first launch does.
 */
ar_status ar_bank_create(ar_bank **out, int64_t T, int32_t d, int32_t r, int32_t capacity,
                         ar_dtype dtype, ar_norm norm, float eps, void *rows,
                         float *inv_rms, float *grad);

/* Release the handle (not the caller's buffers). NULL is accepted. */
ar_status ar_bank_destroy(ar_bank *bank);

/* Rows appended so far. */
ar_status ar_bank_row_count(const ar_bank *bank, int32_t *count);

/* Device address of row `row` (0 <= row < capacity): lets a producer write
 * its sublayer output straight into the next bank slot (then append it with
 * src = that address, which copies nothing). */
ar_status ar_bank_row_ptr(const ar_bank *bank, int32_t row, void **ptr);

/*
 * Append one source row (MHAR Sec. 2.2: after the embedding, every attention
 * and every MLP sublayer contributes its output, unnormalised, as one source;
 * LR-AttnRes Eq. 5-6 and Figure 11 for the block variant) and cache its per-token inverse RMS once, for reuse by
 * every later site.
 *   src             : device [T, d] of the bank dtype. It may be the address
 *                     of the slot being filled (ar_bank_row_ptr), then
 *                     nothing is copied.
 *   accumulate_from : -1 to store src as is; otherwise a row index p already
 *                     appended: the new row is rows[p] + src computed in fp32
 *                     and rounded once to the storage dtype (a new immutable
 *                     partial-sum version; LR-AttnRes Sec. 3.3: the block
 *                     sum is formed at full width before any key is sliced
 *                     out of it or normalised).
 *   out_row         : receives the new row's index (may be NULL).
 * Errors: AR_ERR_CAPACITY (bank full), AR_ERR_INVALID_ARG (bad p, null src),
 * AR_ERR_ALIGN, AR_ERR_CUDA.
 */
ar_status ar_bank_append(ar_bank *bank, const void *src, int32_t accumulate_from,
                         int32_t *out_row, void *stream);

/*
 * ar_bank_append for a strided source: element (t, c) of the [T, d] source
 * is src[t * token_stride + c * elem_stride] ("Low-Rank Attention
 * Residuals", Appendix I: the operator is checked on strided sources). The
 * stored row, its inverse RMS and everything downstream are bit for bit those
 * of ar_bank_append on a contiguous copy of the same values.
 *   token_stride : elements between tokens (>= 0; 0 repeats one row)
 *   elem_stride  : elements between coordinates (>= 1)
 * src needs only the alignment of one element; a contiguous source with
 * 16-byte aligned token rows takes 16-byte accesses, any other one element at
 * a time. Errors: as ar_bank_append; AR_ERR_INVALID_ARG for negative strides.
 */
ar_status ar_bank_append_strided(ar_bank *bank, const void *src, int64_t token_stride,
                                 int64_t elem_stride, int32_t accumulate_from, int32_t *out_row,
                                 void *stream);

/* Start a new backward pass: mark every gradient row untouched, so that the
 * first backward that reaches a row stores into it and later ones accumulate
 * (MHAR Appendix E, FIRST_CALL). No memset is issued. */
ar_status ar_bank_zero_grad(ar_bank *bank);

/* Forget all rows, routing records and gradient flags (next microbatch). */
ar_status ar_bank_reset(ar_bank *bank);

/*
 * Forward of one routing site: online softmax over the listed sources with
 * the RMSNorm key computed in the same pass (MHAR Appendix E, forward kernel,
 * Figure 9), each source row read once.
 *   rows, n_src : host int32 list of appended rows, 1..AR_MAX_SOURCES entries.
 *                 A row may be listed more than once: the softmax runs over
 *                 the list, so a row listed k times carries k times the
 *                 weight of one listed once. It is still read once per token
 *                 (log k is added to its score) and its gradient is the sum
 *                 over its k entries. Such sites run on the scalar-access
 *                 kernels (see "Shapes" above).
 *   H           : routing heads
 *   q           : device float [r], the site's query
 *   g           : device float [r] RMSNorm weight, or NULL for ones
 *   out         : device [T, d] of the bank dtype
 *   lse         : device float [T, H], per-head log-sum-exp (natural log)
 *   site_id     : caller's id of this site; pushed on the bank's call record
 *                 so that the backward can check reverse order.
 * Errors: AR_ERR_INVALID_ARG (row not appended, n_src out of range, null
 * pointers), AR_ERR_SHAPE (d % H or r % H nonzero),
 * AR_ERR_UNSUPPORTED, AR_ERR_ALIGN, AR_ERR_CUDA.
 */
ar_status ar_route_fwd(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                       const float *q, const float *g, void *out, float *lse,
                       int32_t site_id, void *stream);

/*
 * ar_bank_append followed by ar_route_fwd, in one call: append src as the
 * next row (rows[accumulate_from] + src when accumulate_from >= 0), then read
 * the site over `rows`, which may list the new row (its index is the bank's
 * row count before the call; it is also returned in *out_row when out_row is
 * not NULL). The forward itself forms the new row (a copy, or the partial sum
 * rounded once, written to the row's slot) and computes its inverse RMS
 * ("Low-Rank Attention Residuals" Eq. 11) from the staged values when the
 * site lists the new row once and runs on
 *   - the four-warp kernels (d a multiple of 1024; src 16-byte aligned
 *     unless it is the slot itself), or
 *   - the one-warp full-key kernels with rows up to 1024 wide (d = 256, 512,
 *     768 or 1024, H a power of two up to 32), when src already sits in its
 *     slot (the pointer ar_bank_row_ptr gives, accumulate_from = -1):
 * one launch instead of two, and the new row is not read back. Otherwise the
 * two calls run one after the other. *fused (when not NULL) is set to 1 in
 * the first case and to 0 in the second. The bank row and its cached inverse
 * RMS are those ar_bank_append gives (the row bit for bit).
 * Arguments as ar_bank_append and ar_route_fwd; the site's checks run before
 * anything is appended, so on an argument error the bank is unchanged.
 * Errors: those of ar_bank_append and ar_route_fwd.
 */
ar_status ar_route_fwd_append(ar_bank *bank, const void *src, int32_t accumulate_from,
                              int32_t *out_row, const int32_t *rows, int32_t n_src, int32_t H,
                              const float *q, const float *g, void *out, float *lse,
                              int32_t site_id, int32_t *fused, void *stream);

/*
 * Forward of one routing site in the delta form of attention residuals:
 *   out = partial + alpha * routed,   routed = the read of ar_route_fwd
 * ("Multi-Head Attention Residuals", Sec. 3.3 "Identity-preserving
 * conversion": h = partial + alpha * routed with a zero-initialised gate, so
 * that alpha = 0 leaves the residual stream untouched; Appendix E, Figure 9:
 * in the delta form the forward's epilogue sums the partial and the gated
 * mix).
 *   partial : device [T, d] of the bank dtype, the intact residual stream
 *   alpha   : device float, the site's gate
 *   out     : device [T, d] of the bank dtype (may not alias partial)
 *   routed  : device [T, d] of the bank dtype; receives the routed mix, which
 *             the backward needs
 *   other arguments as ar_route_fwd. In the pages' mid-training setup the
 *   sources are a per-call stack: a learnable null source
 *   (ar_bank_append_broadcast) plus one delta per block.
 * Errors: as ar_route_fwd; AR_ERR_INVALID_ARG for a null partial, alpha or
 * routed; AR_ERR_UNSUPPORTED for shapes served by the one-warp sliced-key
 * kernels (r < d with d not a multiple of 1024).
 */
ar_status ar_route_fwd_delta(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                             const float *q, const float *g, const void *partial,
                             const float *alpha, void *out, void *routed, float *lse,
                             int32_t site_id, void *stream);

/*
 * A routing site with its query and norm weight given as strided vectors
 * ("Low-Rank Attention Residuals", Appendix I: the operator is checked on
 * strided queries), e.g. one column of a [r, sites] parameter matrix.
 *   rows, n_src, H, site_id : as in ar_route_fwd
 *   q, q_stride : device float, entry c at q[c * q_stride] (q_stride >= 1)
 *   g, g_stride : the same for g, or g = NULL for ones
 * In the backward, dq is written with q's stride and dg with g's stride (the
 * gradient laid out like its parameter).
 */
typedef struct ar_site {
    const int32_t *rows;
    int32_t n_src;
    int32_t H;
    const float *q;
    int64_t q_stride;
    const float *g;
    int64_t g_stride;
    int32_t site_id;
} ar_site;

/* Forward of one site described by an ar_site. partial, alpha and routed are
 * all NULL (plain read, as ar_route_fwd) or all non-NULL (delta form, as
 * ar_route_fwd_delta). Errors: as those calls; AR_ERR_INVALID_ARG for a
 * NULL site, a stride < 1, or a partial set of the delta pointers. */
ar_status ar_route_fwd_site(ar_bank *bank, const ar_site *site, const void *partial,
                            const float *alpha, void *out, void *routed, float *lse,
                            void *stream);

/* Bytes of device workspace ar_route_bwd (and ar_route_bwd_delta) needs for
 * this bank and H: per-warp (or per-block) partial sums of dq/dg and of
 * dL/dalpha. Depends on the current device. */
ar_status ar_route_bwd_workspace(const ar_bank *bank, int32_t H, size_t *bytes);

/*
 * Backward of one routing site (MHAR Appendix E, backward kernel: a single
 * launch that recomputes the key norms and adds into the gradient rows,
 * Figure 10; the value/routing split of LR-AttnRes Eq. 15 with the score
 * gradient of Eq. 21/22). Given dL/dout it emits dL/ds_n for every listed source into the
 * bank's fp32 gradient rows — a store on a row's first touch since
 * ar_bank_zero_grad, an in-place accumulation afterwards — and dL/dq, dL/dg.
 *   rows, n_src, H, q, g : exactly as in the forward of this site
 *   out   : device [T, d], this site's forward output (its per-head dot with
 *           dout is the softmax coupling term). The coupling is read from
 *           this output as stored, in one pass, where MHAR Figure 10 sums it
 *           over the sources in a first pass: with a bf16 bank its rounding
 *           enters every routing feedback as w * <dout_h, rounding_h>. That is
 *           small, but a source that holds nearly all of a head's weight has
 *           a nearly cancelling feedback. Its key-path gradient can then
 *           differ from the exact one by a few percent of the row's largest
 *           gradient: 3.3 % measured on the LR page's 4B shape with peaked
 *           queries. ar_route_bwd_exact sums the coupling over the sources
 *           instead.
 *   dout  : device [T, d] of the bank dtype, dL/dout
 *   lse   : device float [T, H] written by this site's forward
 *   dq    : device float [r], overwritten with dL/dq
 *   dg    : device float [r] overwritten with dL/dg, or NULL to skip
 *   ws    : device workspace of ws_bytes >= ar_route_bwd_workspace()
 *   site_id: must equal the most recent forward's site_id not yet
 *           backpropagated (reverse forward order, MHAR Appendix E);
 *           otherwise AR_ERR_ORDER and nothing runs.
 * Errors: as the forward, plus AR_ERR_ORDER, AR_ERR_CAPACITY (workspace too
 * small), AR_ERR_INVALID_ARG (bank created without grad).
 */
ar_status ar_route_bwd(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                       const float *q, const float *g, const void *out, const void *dout,
                       const float *lse, float *dq, float *dg, void *ws, size_t ws_bytes,
                       int32_t site_id, void *stream);

/*
 * Fold one gradient row into another: grad[dst_row] += grad[src_row] over all
 * T x d entries (fp32). A row that has not been written since
 * ar_bank_zero_grad counts as zero, and dst_row is marked written.
 * Use: block partial sums are stored as versions, row t+1 = row t + o_{t+1};
 * version t+1's adjoint reaches version t (and so every write of the block)
 * through this fold, run after the backward of every site that reads row
 * t+1 ("Low-Rank Attention Residuals", Appendix B.4: every write of a block
 * receives the adjoint of the block sum; Figure 11's partial += y).
 * Errors: AR_ERR_INVALID_ARG (rows not appended, equal rows, bank without
 * gradient rows), AR_ERR_CUDA.
 */
ar_status ar_bank_grad_fold(ar_bank *bank, int32_t dst_row, int32_t src_row, void *stream);

/*
 * Reads of up to AR_MAX_QUERIES sites over one source list, in one pass over
 * the sources: phase 1 of two-phase block inference ("Low-Rank Attention
 * Residuals", Sec. 3.4: the queries are input-independent, so the inter-block
 * reads of all sites of a block can be done first, together; each site's
 * intra-block read is merged in later with ar_route_merge). Output i is
 * what ar_route_fwd would give with query q[i] and norm weight g[i], while
 * every row is read once per token instead of n_q times.
 *   rows, n_src, H : as ar_route_fwd (a row listed twice enters once with
 *                    log 2 added to its score)
 *   n_q            : number of queries, 1..AR_MAX_QUERIES
 *   q, g           : host arrays of n_q device pointers to float [r]
 *                    (contiguous); g may be NULL (ones everywhere), and so may
 *                    any g[i]
 *   out, lse       : host arrays of n_q device pointers: out[i] [T, d] of the
 *                    bank dtype (16-byte aligned), lse[i] float [T, H]
 * Forward only: nothing enters the bank's call record, and there is no
 * backward (inference). Shapes: d a multiple of 256 up to 4096, d/H and r/H
 * multiples of 8, r <= 2048, and a token's n_src rows (n_src * d * dtype
 * bytes) within about 200 KB of shared memory; others get
 * AR_ERR_UNSUPPORTED (the per-site ar_route_fwd serves every shape). Each
 * block stages all rows of a token at once, computes every query's scores
 * and weights, then sums the rows per column for every query.
 * Errors: AR_ERR_INVALID_ARG (rows, n_q out of range, null pointers),
 * AR_ERR_SHAPE, AR_ERR_UNSUPPORTED, AR_ERR_ALIGN, AR_ERR_CUDA.
 */
ar_status ar_route_fwd_multi(const ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                             int32_t n_q, const float *const *q, const float *const *g,
                             void *const *out, float *const *lse, void *stream);

/*
 * Merge two partial reads of one site over disjoint source sets A and B into
 * the read over A u B, per head, by the online-softmax update:
 *   lse = log(e^lse_A + e^lse_B),
 *   out = e^(lse_A - lse) out_A + e^(lse_B - lse) out_B   on the head's slice.
 * This is the merge of two-phase block inference ("Low-Rank Attention
 * Residuals", Sec. 3.4: input-independent queries let the inter-block reads
 * of a whole block be done first; each site's intra-block read is merged in).
 *   out_a, out_b, out : device [T, d] of the bank dtype (out may alias either)
 *   lse_a, lse_b, lse : device float [T, H] (lse may alias either)
 * The bank supplies T, d and the dtype only. Errors: AR_ERR_INVALID_ARG,
 * AR_ERR_SHAPE (d % H), AR_ERR_ALIGN, AR_ERR_CUDA.
 */
ar_status ar_route_merge(const ar_bank *bank, int32_t H, const void *out_a, const float *lse_a,
                         const void *out_b, const float *lse_b, void *out, float *lse, void *stream);

/*
 * Block schedule of LR-AttnRes (Figure 11): M sublayers in NB blocks whose
 * last sublayers are ceil(M*j/NB); NB <= 0 or NB >= M means full routing.
 * Bank row 0 is the embedding; row t (1..M) is the partial sum after
 * sublayer t. Outputs (host arrays):
 *   acc_from  [M+1] : -1 if row t is stored as is (row 0, or the first
 *                     sublayer of a block), else the row it accumulates onto
 *   site_ptr  [M+2] : CSR offsets; site t (0..M) reads
 *                     site_rows[site_ptr[t] .. site_ptr[t+1])
 *   site_rows [cap] : row lists; *site_rows_len receives the total length
 * Errors: AR_ERR_INVALID_ARG (M < 1, null outputs), AR_ERR_CAPACITY
 * (site_rows_cap too small; *site_rows_len still receives the need).
 */
ar_status ar_block_schedule(int32_t M, int32_t NB, int32_t *acc_from, int32_t *site_ptr,
                            int32_t *site_rows, int64_t site_rows_cap, int64_t *site_rows_len);

/*
 * Backward of ar_route_fwd_delta. With G = dL/dout: the routed mix receives
 * alpha * G, so the source gradients, dq and dg are those of ar_route_bwd for
 * upstream gradient alpha * G; dL/dalpha = sum over tokens of <G, routed>; and
 * dL/dpartial = G (the caller uses dout directly, nothing is computed).
 *   routed : device [T, d], written by this site's forward
 *   alpha  : device float, the gate the forward used
 *   dalpha : device float, overwritten with dL/dalpha
 *   other arguments as ar_route_bwd (same workspace size). In the pages'
 *   per-call form every call owns fresh gradient rows: call ar_bank_zero_grad
 *   (or use a bank per call) before it, so that every row is stored, not
 *   accumulated.
 * Errors: as ar_route_bwd; AR_ERR_INVALID_ARG for a null alpha or dalpha.
 */
ar_status ar_route_bwd_delta(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                             const float *q, const float *g, const void *routed,
                             const void *dout, const float *lse, const float *alpha, float *dq,
                             float *dg, float *dalpha, void *ws, size_t ws_bytes, int32_t site_id,
                             void *stream);

/* Backward of one site described by an ar_site. alpha and dalpha are both
 * NULL (as ar_route_bwd; `out` is the forward output) or both non-NULL (as
 * ar_route_bwd_delta; `out` is the routed mix). dq is written with the
 * site's q_stride, dg with its g_stride. Errors: as those calls;
 * AR_ERR_INVALID_ARG for a NULL site, a stride < 1, or only one of
 * alpha/dalpha. */
ar_status ar_route_bwd_site(ar_bank *bank, const ar_site *site, const void *out,
                            const void *dout, const float *lse, const float *alpha, float *dq,
                            float *dg, float *dalpha, void *ws, size_t ws_bytes, void *stream);

/* ar_route_bwd_site (plain form) with the coupling term summed over the
 * sources, as in the first pass of "Multi-Head Attention Residuals", Appendix E
 * (Figure 10):
 *   coupling[t, h] = sum_n w_{n,h} <dout_[h], s_{n,[h]}>
 * is computed into `coupling` first (one more read of the site's rows), and
 * the backward then uses it in place of the per-head dot of dout with `out`. This makes the source, query and norm-weight
 * gradients exact up to fp32 rounding, whatever the precision of the stored
 * forward output. For a bf16 bank, the one-pass backward (ar_route_bwd and
 * ar_route_bwd_site) carries the output's rounding into the feedback of a
 * dominant source (see ar_route_bwd, `out`). `out` is still read (the token
 * buffers).
 *   coupling : device float [T, H], written (caller-owned scratch)
 *   alpha, dalpha : must be NULL (the delta form is not served here)
 *   other arguments as ar_route_bwd_site.
 * Errors: as ar_route_bwd_site; AR_ERR_UNSUPPORTED for a non-NULL alpha or
 * dalpha, AR_ERR_INVALID_ARG for a NULL coupling when T > 0, AR_ERR_ALIGN for
 * one not 4-byte aligned. */
ar_status ar_route_bwd_exact(ar_bank *bank, const ar_site *site, const void *out,
                             const void *dout, const float *lse, const float *alpha,
                             float *coupling, float *dq, float *dg, float *dalpha, void *ws,
                             size_t ws_bytes, void *stream);

/*
 * Append a row that holds the same vector for every token (the learnable null
 * source of the delta form, "Multi-Head Attention Residuals", Sec. 3.3), and
 * cache its inverse RMS.
 *   vec : device [d] of the bank dtype. Errors as ar_bank_append.
 */
ar_status ar_bank_append_broadcast(ar_bank *bank, const void *vec, int32_t *out_row, void *stream);

/*
 * out[c] = sum over tokens of the gradient row `row` (the gradient of a
 * broadcast source such as the null source), in a fixed summation order.
 *   out : device float [d], overwritten (zeros if the row was not written
 *         since ar_bank_zero_grad). Errors: AR_ERR_INVALID_ARG, AR_ERR_ALIGN,
 *         AR_ERR_CUDA.
 */
ar_status ar_bank_grad_token_sum(const ar_bank *bank, int32_t row, float *out, void *stream);

/*
 * ar_route_bwd_noalloc: ar_route_bwd with no caller workspace. There is no
 * counterpart in the papers; this entry point exists for callers that cannot
 * allocate device memory (for example an engine plugin whose execute hook may
 * not call cudaMalloc, or code embedded in a process whose device memory
 * belongs to another framework's pool).
 *   Arguments, results and checks are those of ar_route_bwd, minus ws and
 *   ws_bytes: the backward's scratch (its per-block dq/dg partial sums) lives
 *   in a fixed device array inside this library, AR_NOALLOC_SCRATCH_BYTES
 *   large (ar_noalloc_scratch_bytes() reports it), which every GPU on which
 *   the library's device code is loaded holds until the process exits. Under
 *   CUDA's lazy module loading (the default) that happens when the library is
 *   first used on the device, which may be this entry point's first call:
 *   count the array against a fixed memory budget from that call on. The
 *   call allocates nothing.
 *   - If ar_route_bwd_workspace() for this bank and H exceeds
 *     AR_NOALLOC_SCRATCH_BYTES, the call returns AR_ERR_CAPACITY and runs
 *     nothing; use ar_route_bwd with a workspace instead.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current, for devices 0..63; a higher
 *     device number gets AR_ERR_CUDA); make that first call before any
 *     stream capture. The address is kept for the life of the process: do not
 *     call cudaDeviceReset on a device between uses of this entry point (the
 *     reset unloads the library's device code, and the kept address would no
 *     longer be valid).
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero). Calls whose kernels can overlap
 *     on the GPU (unordered streams) race on it: serialise them.
 */
#define AR_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
ar_status ar_route_bwd_noalloc(ar_bank *bank, const int32_t *rows, int32_t n_src, int32_t H,
                               const float *q, const float *g, const void *out, const void *dout,
                               const float *lse, float *dq, float *dg, int32_t site_id,
                               void *stream);

/* The size of ar_route_bwd_noalloc's fixed scratch array in bytes
 * (AR_NOALLOC_SCRATCH_BYTES, the value the library was compiled with). */
ar_status ar_noalloc_scratch_bytes(size_t *bytes);

/* Read and clear the device error word of the current device (bit mask of
 * AR_DEVERR_*; 0 = none). This call synchronises the device. */
ar_status ar_device_error(uint32_t *bits);

/* The device error word as a status: synchronises the device, reads and
 * clears the word, and returns AR_ERR_BOUNDS if a checked kernel skipped an
 * access since the last read (AR_DEVERR_BOUNDS), else AR_ERR_TIMEOUT if a
 * device-side wait ran out (AR_DEVERR_WAIT_TIMEOUT), AR_OK if neither
 * happened, AR_ERR_CUDA if the device could not be read. */
ar_status ar_device_status(void);

/*
 * Test of the failure path (no counterpart in the papers): the forward of a
 * site, as ar_route_fwd, except that every shared-memory stage is armed for
 * its row's bytes and no copy is ever issued. Each warp's first wait then
 * runs out after poll_limit polls with nothing in flight; the kernel sets
 * AR_DEVERR_WAIT_TIMEOUT in the device error word, waits at most poll_limit
 * polls per armed stage, and returns without writing out or lse. The host
 * sees it through ar_device_status() (AR_ERR_TIMEOUT); the context stays
 * usable. Nothing is recorded in the bank (no backward may follow).
 *   Served on the one-warp full-key forward only: r = d, d a multiple of 256
 *   from 768 to 2048 (or 256 and 512 with H > 4), H a power of two <= 32,
 *   distinct rows; other shapes get AR_ERR_UNSUPPORTED. poll_limit >= 1 and
 *   T >= 1 (else AR_ERR_INVALID_ARG). Other checks as ar_route_fwd.
 */
ar_status ar_route_fwd_lost_copies(ar_bank *bank, const int32_t *rows, int32_t n_src,
                                   int32_t H, const float *q, const float *g, void *out,
                                   float *lse, uint32_t poll_limit, void *stream);

/*
 * Range checks (a debugging aid with no counterpart in the papers; it stands
 * in for a memory checker). A library built with AR_CHECKED defined
 * (libattnres_gb300_checked.so) gives every kernel launch a table of the
 * buffers of its launch: the bank's rows and gradient rows, where an access
 * must fall inside one row that the site lists (a store into the bank only
 * inside the row the call appends), and every other buffer the call takes,
 * read-only where the call only reads it, with the extents stated in this
 * header. Each global access the kernels make through their load, store and
 * bulk-copy paths, and each access to the rows staged in shared memory
 * (not the tensor-core tile loads), is checked for range and alignment
 * first. An access that fails is not made (a load gives
 * zeros, a bulk copy completes its bytes on its mbarrier without copying),
 * the first one is recorded, and AR_DEVERR_BOUNDS is set in the device error
 * word. Nothing traps. Every kernel of the library is checked, the append,
 * merge, token-sum, gradient-fold and dq/dg reduction kernels included.
 *
 * ar_checked_fault: *checked = 1 in a checked library, else 0. In a checked
 * library it synchronises the device and returns the first failed access
 * since the last call: *addr (a global address, or the shared-window offset
 * for kind 3), *bytes, *kind (0 none, 1 global load, 2 global store,
 * 3 shared memory), then clears the record. In an unchecked library the
 * outputs are zero and nothing touches the device. Errors:
 * AR_ERR_INVALID_ARG (a null pointer), AR_ERR_CUDA.
 *
 * ar_checked_trim_out: a test of the checks themselves. The next launches
 * declare the output buffer out of a forward or a merge (each out[i] of a
 * multi-query read) `bytes` shorter than the call states, so that stores
 * into its tail are refused although they lie inside the real buffer; 0
 * restores the stated extents. Host state of the library,
 * not thread-safe. AR_ERR_UNSUPPORTED in an unchecked library,
 * AR_ERR_INVALID_ARG for a negative size.
 */
ar_status ar_checked_fault(int32_t *checked, uint64_t *addr, uint32_t *bytes, uint32_t *kind);
ar_status ar_checked_trim_out(int64_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H */

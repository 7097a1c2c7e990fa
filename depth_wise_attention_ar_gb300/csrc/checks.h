// Range-check decisions of the checked build (AR_CHECKED), shared by the
// device checks in common.cuh and a host test: may an access of `bytes` bytes
// at global address x (a load or a store, `align`-byte aligned) be made under
// a launch's buffer table?
//   - x and bytes are multiples of align;
//   - inside the bank or the gradient rows ([cap, T, d] row arrays) it lies
//     within one row, which the launch lists: in the bank a store only into
//     the row the call appends (rows[fresh1 - 1]), and a load also from the
//     row a partial sum starts from (acc_row);
//   - elsewhere it lies within one span of the table, a writable one for a
//     store.
#pragma once

#include <stdint.h>

#include "ar_internal.h"

#ifdef AR_CHECKED
#ifdef __CUDACC__
#define AR_HD __host__ __device__
#else
#define AR_HD
#endif

namespace ar {

AR_HD inline bool chk_row_ok(const RouteArgs &a, uint64_t row, bool bank, bool store)
{
    if (bank && store) return a.fresh1 > 0 && row == static_cast<uint64_t>(a.rows[a.fresh1 - 1]);
    for (int i = 0; i < a.n_src; ++i)
        if (row == static_cast<uint64_t>(a.rows[i])) return true;
    return bank && a.fresh1 > 0 && a.acc_row >= 0 && row == static_cast<uint64_t>(a.acc_row);
}

AR_HD inline bool chk_decide(const RouteArgs &a, uint64_t x, uint32_t bytes, bool store,
                             uint32_t align)
{
    const CheckTable &c = a.chk;
    const uint64_t e = x + bytes;
    if ((x | bytes) % align != 0) return false;
    for (int b = 0; b < 2; ++b) {
        const uint64_t base = b ? c.grad : c.bank, rb = b ? c.grad_row : c.bank_row;
        if (base && rb && x >= base && x < base + static_cast<uint64_t>(c.cap) * rb) {
            const uint64_t row = (x - base) / rb;
            return e <= base + (row + 1) * rb && chk_row_ok(a, row, b == 0, store);
        }
    }
    for (int i = 0; i < c.n; ++i)
        if (x >= c.lo[i] && e <= c.hi[i] && (!store || c.wr[i])) return true;
    return false;
}

}  // namespace ar

#undef AR_HD
#endif

// Host test of the range-check decisions of the checked build (chk_decide in
// depth_wise_attention_ar_gb300/csrc/checks.h): a fabricated buffer table and
// accesses at its edges. Prints one line per failed case, then "checked N
// cases, F failed"; exits non-zero when any case fails.
#include <cstdio>
#include <cstring>

#include "checks.h"

using ar::RouteArgs;

static int g_cases = 0, g_failed = 0;

static void expect(const char *what, bool got, bool want)
{
    ++g_cases;
    if (got != want) {
        ++g_failed;
        std::printf("FAIL %s: got %d, want %d\n", what, (int)got, (int)want);
    }
}

static void span(RouteArgs &a, uint64_t lo, uint64_t bytes, bool wr)
{
    ar::CheckTable &c = a.chk;
    c.lo[c.n] = lo;
    c.hi[c.n] = lo + bytes;
    c.wr[c.n] = wr ? 1 : 0;
    ++c.n;
}

int main()
{
    // bank: 6 rows of 4096 bytes at 0x100000; gradient rows: 6 rows of 8192
    // bytes at 0x200000; spans: a read-only one at 0x300000 (1024 bytes) and
    // a writable one at 0x400000 (512 bytes)
    static RouteArgs a;
    std::memset(&a, 0, sizeof(a));
    ar::CheckTable &c = a.chk;
    c.bank = 0x100000;
    c.bank_row = 4096;
    c.grad = 0x200000;
    c.grad_row = 8192;
    c.cap = 6;
    a.n_src = 2;
    a.rows[0] = 1;
    a.rows[1] = 4;
    a.acc_row = -1;
    span(a, 0x300000, 1024, false);
    span(a, 0x400000, 512, true);
    const uint64_t B = 0x100000, G = 0x200000;

    // bank rows
    expect("load inside a listed row", ar::chk_decide(a, B + 4096 + 32, 16, false, 16), true);
    expect("load at the end of a listed row", ar::chk_decide(a, B + 2 * 4096 - 16, 16, false, 16), true);
    expect("load of a row not listed", ar::chk_decide(a, B + 2 * 4096, 16, false, 16), false);
    expect("load of row 0, not listed", ar::chk_decide(a, B, 16, false, 16), false);
    expect("load straddling into the next row", ar::chk_decide(a, B + 2 * 4096 - 16, 32, false, 16), false);
    expect("store into a listed row without an append", ar::chk_decide(a, B + 4096, 16, true, 16), false);
    expect("load past the last row", ar::chk_decide(a, B + 6 * 4096, 16, false, 16), false);
    // the append of row 4 (second in the list), formed from row 3
    a.fresh1 = 2;
    a.acc_row = 3;
    expect("store into the appended row", ar::chk_decide(a, B + 4 * 4096 + 64, 16, true, 16), true);
    expect("store into another listed row", ar::chk_decide(a, B + 1 * 4096 + 64, 16, true, 16), false);
    expect("load of the partial sum's first row", ar::chk_decide(a, B + 3 * 4096, 16, false, 16), true);
    expect("store into the partial sum's first row", ar::chk_decide(a, B + 3 * 4096, 16, true, 16), false);
    a.fresh1 = 0;
    expect("load of acc_row without an append", ar::chk_decide(a, B + 3 * 4096, 16, false, 16), false);
    a.acc_row = -1;

    // gradient rows: loads and stores of listed rows only
    expect("gradient store, listed row", ar::chk_decide(a, G + 4 * 8192 + 32, 32, true, 32), true);
    expect("gradient load, listed row", ar::chk_decide(a, G + 1 * 8192, 32, false, 16), true);
    expect("gradient store, row not listed", ar::chk_decide(a, G + 2 * 8192, 32, true, 32), false);
    expect("gradient store straddling two rows", ar::chk_decide(a, G + 2 * 8192 - 16, 32, true, 16), false);

    // spans
    expect("load in the read-only span", ar::chk_decide(a, 0x300000 + 1008, 16, false, 16), true);
    expect("load past the read-only span", ar::chk_decide(a, 0x300000 + 1024, 16, false, 16), false);
    expect("load overlapping its end", ar::chk_decide(a, 0x300000 + 1016, 16, false, 8), false);
    expect("store into the read-only span", ar::chk_decide(a, 0x300000, 4, true, 4), false);
    expect("store into the writable span", ar::chk_decide(a, 0x400000 + 508, 4, true, 4), true);
    expect("store past the writable span", ar::chk_decide(a, 0x400000 + 512, 4, true, 4), false);
    expect("store before the writable span", ar::chk_decide(a, 0x400000 - 4, 4, true, 4), false);
    expect("address in no buffer", ar::chk_decide(a, 0x500000, 4, false, 4), false);

    // alignment
    expect("16-byte access at an 8-byte boundary", ar::chk_decide(a, B + 4096 + 8, 16, false, 16), false);
    expect("32-byte store at a 16-byte boundary", ar::chk_decide(a, G + 8192 + 16, 32, true, 32), false);
    expect("size not a multiple of the alignment", ar::chk_decide(a, 0x300000, 24, false, 16), false);
    expect("2-byte element at an odd address", ar::chk_decide(a, 0x300001, 2, false, 2), false);
    expect("2-byte element at an even address", ar::chk_decide(a, 0x300002, 2, false, 2), true);

    // no bank or gradient structure: only spans count
    c.bank = 0;
    c.grad = 0;
    expect("bank address without bank rows", ar::chk_decide(a, B + 4096, 16, false, 16), false);
    span(a, B, 6 * 4096, false);
    expect("bank address in a plain span", ar::chk_decide(a, B + 2 * 4096, 16, false, 16), true);

    std::printf("checked %d cases, %d failed\n", g_cases, g_failed);
    return g_failed ? 1 : 0;
}

"""Two-phase block inference ("Low-Rank Attention Residuals", Sec. 3.4): each
site's read is split into the inter-block part (embedding + completed block
sums, all available when the block starts) and the intra-block part (the
current partial sum); ar_route_merge combines the two by their per-head
log-sum-exp. The merged read must equal the oracle's read over all the site's
sources."""

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from depth_wise_attention_ar_gb300 import build
    build.build()
    from depth_wise_attention_ar_gb300 import binding
    return binding


def _t64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def _nmax(x, ref):
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.mark.parametrize("d,r,H,dtype", [(512, 512, 4, "f32"), (1024, 256, 4, "bf16"),
                                         (4096, 1024, 8, "bf16")])
def test_two_phase_block_read_equals_single_read(B, orc, d, r, H, dtype):
    import torch
    from oracle import schedule, storage
    T, M, NB = 200, 12, 3
    acc, sites = B.ar_block_schedule(M, NB)
    inp = synth.HostInputs(seed=17, q_std=0.8, g_kind="random")
    bank = B.Bank(T, d, r, M + 1, dtype)
    for t in range(M + 1):
        o = inp.output(t, T, d, dtype)
        if acc[t] < 0:
            bank.rows[t].copy_(o)
            bank.append(bank.rows[t])
        else:
            bank.append(o, acc[t])
    ref_rows = storage.block_bank([inp.host_output(t, T, d, dtype) for t in range(M + 1)],
                                  schedule.block_plan(M, NB), dtype)
    tol = 1e-5 if dtype == "f32" else 2e-2
    checked = 0
    for t in range(1, M + 1):
        rows = sites[t]
        if t in schedule.block_ends(M, NB):
            continue              # right after a block end there is no partial sum
        inter, partial = rows[:-1], rows[-1]
        q, g = inp.query(t, r), inp.norm_weight(t, r)
        out_a, lse_a = bank.route_fwd(inter, H, q, g, site_id=t)
        out_b, lse_b = bank.route_fwd([partial], H, q, g, site_id=t)
        out = torch.empty_like(out_a)
        lse = torch.empty_like(lse_a)
        B.ar_route_merge(bank.handle, H, out_a, lse_a, out_b, lse_b, out, lse)
        torch.cuda.synchronize()
        ref_out, ref_lse = orc.route_fwd([ref_rows[j] for j in rows], inp.host_query(t, r),
                                         inp.host_norm_weight(t, r), H, r=r)
        assert _nmax(_t64(out), ref_out) < tol, t
        assert _nmax(_t64(lse), ref_lse) < tol, t
        checked += 1
    assert checked >= 6


@pytest.mark.parametrize("d,r,H,dtype,nq,N", [(4096, 1024, 8, "bf16", 8, 9), (1280, 1280, 8, "bf16", 3, 5),
                                               (512, 512, 4, "f32", 1, 4), (1536, 384, 1, "f32", 8, 9),
                                               (2048, 512, 4, "f32", 5, 7), (768, 768, 3, "bf16", 2, 3)])
def test_multi_query_read_equals_per_query_reads(B, orc, d, r, H, dtype, nq, N):
    """ar_route_fwd_multi: output i and lse i match the oracle's read with
    query i, for full and sliced keys and 1 to 8 queries."""
    import torch
    T = 157
    inp = synth.HostInputs(seed=31, q_std=0.8, g_kind="random")
    bank = B.Bank(T, d, r, N, dtype)
    for j in range(N):
        bank.append(inp.output(j, T, d, dtype))
    rows = list(range(N))
    qs = [inp.query(100 + i, r) for i in range(nq)]
    gs = [inp.norm_weight(100 + i, r) if i % 2 == 0 else None for i in range(nq)]
    outs, lses = bank.route_fwd_multi(rows, H, qs, gs)
    torch.cuda.synchronize()
    assert B.ar_device_error() == 0
    srcs = [inp.host_output(j, T, d, dtype) for j in range(N)]
    tol = 1e-5 if dtype == "f32" else 2e-2
    for i in range(nq):
        gh = inp.host_norm_weight(100 + i, r) if gs[i] is not None else None
        ref_out, ref_lse = orc.route_fwd(srcs, inp.host_query(100 + i, r), gh, H, r=r)
        assert _nmax(_t64(outs[i]), ref_out) < tol, i
        assert _nmax(_t64(lses[i]), ref_lse) < tol, i


@pytest.mark.parametrize("d,r,H,nq,rows,T", [
    (4096, 2048, 8, 8, list(range(16)), 131),    # 16 rows: the ring only fits one block per SM
    (4096, 1024, 8, 1, list(range(16)), 100),    # one query, fewer tokens than blocks
    (4096, 1024, 8, 4, [0, 1, 2, 1, 3], 157),    # a row listed twice
    (2304, 1152, 8, 8, list(range(9)), 157),     # 256-column tiles, heads across 64-column groups
])
def test_multi_query_read_streaming_shapes(B, orc, d, r, H, nq, rows, T):
    """The tiled multi-query kernel at the edges of its layout: the most rows,
    a single query, fewer tokens than blocks, a repeated row (its score gets
    log 2 added), tiles of 256 columns with heads that change inside a 64-column
    group; with 16 rows the ring wraps inside a token. Every output and lse against the
    oracle's read over the listed sources."""
    inp = synth.HostInputs(seed=43, q_std=0.8, g_kind="random")
    nrow = max(rows) + 1
    bank = B.Bank(T, d, r, nrow, "bf16")
    for j in range(nrow):
        bank.append(inp.output(j, T, d, "bf16"))
    qs = [inp.query(200 + i, r) for i in range(nq)]
    gs = [inp.norm_weight(200 + i, r) for i in range(nq)]
    outs, lses = bank.route_fwd_multi(rows, H, qs, gs)
    import torch
    torch.cuda.synchronize()
    assert B.ar_device_error() == 0
    srcs = [inp.host_output(j, T, d, "bf16") for j in rows]
    for i in range(nq):
        ref_out, ref_lse = orc.route_fwd(srcs, inp.host_query(200 + i, r),
                                         inp.host_norm_weight(200 + i, r), H, r=r)
        assert _nmax(_t64(outs[i]), ref_out) < 2e-2, i
        assert _nmax(_t64(lses[i]), ref_lse) < 2e-2, i


@pytest.mark.parametrize("d,r,H,dtype", [(4096, 1024, 8, "bf16"), (1024, 256, 4, "f32")])
def test_two_phase_with_batched_phase_one(B, orc, d, r, H, dtype):
    """Phase 1 reads the inter-block rows once for all the sites of a block
    (ar_route_fwd_multi, the block's input-independent queries); phase 2 reads
    each site's partial sum and merges. Every merged read equals the oracle's
    read over all of the site's sources."""
    import torch
    from oracle import schedule, storage
    T, M, NB = 131, 12, 3
    acc, sites = B.ar_block_schedule(M, NB)
    inp = synth.HostInputs(seed=37, q_std=0.8, g_kind="random")
    bank = B.Bank(T, d, r, M + 1, dtype)
    for t in range(M + 1):
        o = inp.output(t, T, d, dtype)
        if acc[t] < 0:
            bank.rows[t].copy_(o)
            bank.append(bank.rows[t])
        else:
            bank.append(o, acc[t])
    ref_rows = storage.block_bank([inp.host_output(t, T, d, dtype) for t in range(M + 1)],
                                  schedule.block_plan(M, NB), dtype)
    ends = set(schedule.block_ends(M, NB))
    # group the sites that read a partial sum by their inter-block rows
    groups = {}
    for t in range(1, M + 1):
        if t in ends:
            continue
        groups.setdefault(tuple(sites[t][:-1]), []).append(t)
    tol = 1e-5 if dtype == "f32" else 2e-2
    checked = 0
    for inter, members in groups.items():
        for k in range(0, len(members), B.AR_MAX_QUERIES):
            batch = members[k:k + B.AR_MAX_QUERIES]
            qs = [inp.query(t, r) for t in batch]
            gs = [inp.norm_weight(t, r) for t in batch]
            outs_a, lses_a = bank.route_fwd_multi(list(inter), H, qs, gs)
            for t, q, g, out_a, lse_a in zip(batch, qs, gs, outs_a, lses_a):
                out_b, lse_b = bank.route_fwd([sites[t][-1]], H, q, g, site_id=t)
                out = torch.empty_like(out_a)
                lse = torch.empty_like(lse_a)
                B.ar_route_merge(bank.handle, H, out_a, lse_a, out_b, lse_b, out, lse)
                torch.cuda.synchronize()
                ref_out, ref_lse = orc.route_fwd([ref_rows[j] for j in sites[t]],
                                                 inp.host_query(t, r), inp.host_norm_weight(t, r),
                                                 H, r=r)
                assert _nmax(_t64(out), ref_out) < tol, t
                assert _nmax(_t64(lse), ref_lse) < tol, t
                checked += 1
    assert checked >= 6

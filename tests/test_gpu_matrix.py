"""The remaining cases of the LR page's correctness matrix ("Low-Rank Attention
Residuals", Appendix I, numerical correctness: strided sources, strided
queries, changed-input replays), through the C ABI.

Strided inputs must give bit for bit what contiguous copies of the same
values give (the kernels read the same numbers; only the addressing
differs). Replays of one captured CUDA graph with new values in its input
buffers are checked against the oracle each time.
"""

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from depth_wise_attention_ar_gb300 import build
    build.build()
    from depth_wise_attention_ar_gb300 import binding
    return binding


def _nmax(x, ref):
    x, ref = np.asarray(x, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _t64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def _same_bits(a, b):
    import torch
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("d,r,H,dtype", [(1280, 1280, 8, "bf16"), (2048, 512, 4, "f32"),
                                         (513, 513, 1, "bf16"), (4096, 4096, 8, "bf16")])
def test_strided_sources(B, d, r, H, dtype):
    """Sources given as a column slice of a wider tensor (token stride 2d + 8),
    as a transposed view (token stride 1, coordinate stride T), and as a row
    slice with an odd token stride: rows, inverse RMS, and the site's outputs
    and gradients equal those of contiguous appends bit for bit."""
    import torch
    T, n = 129, 4
    inp = synth.HostInputs(seed=21, q_std=0.5, g_kind="random")
    srcs = [inp.output(j, T, d, dtype) for j in range(n)]
    ref = B.Bank(T, d, r, n, dtype)
    got = B.Bank(T, d, r, n, dtype)
    for j, s in enumerate(srcs):
        acc = 2 if j == 3 else -1                   # row 3: a block partial sum on row 2
        ref.append(s, acc)
        if j % 3 == 0:
            wide = torch.zeros((T, 2 * d + 8), dtype=s.dtype, device="cuda")
            wide[:, 8:8 + d] = s
            view = wide[:, 8:8 + d]
        elif j % 3 == 1:
            view = s.t().contiguous().t()
        else:
            wide = torch.zeros((T, d + 1), dtype=s.dtype, device="cuda")
            wide[:, :d] = s
            view = wide[:, :d]
        assert not view.is_contiguous()
        got.append(view, acc)
    torch.cuda.synchronize()
    assert _same_bits(got.rows, ref.rows)
    assert _same_bits(got.inv_rms(), ref.inv_rms())
    rows = [0, 1, 2, 3]
    q, g = inp.query(3, r), inp.norm_weight(3, r)
    res = []
    for bank in (ref, got):
        out, lse = bank.route_fwd(rows, H, q, g, site_id=1)
        bank.zero_grad()
        dq, dg = bank.route_bwd(rows, H, q, g, out, inp.dout(3, T, d, dtype), lse, site_id=1)
        res.append((out, lse, dq, dg, bank.grad))
    torch.cuda.synchronize()
    for a, b in zip(*res):
        assert _same_bits(a, b)


@pytest.mark.parametrize("d,r,H,dtype", [(1280, 1280, 8, "bf16"), (4096, 1024, 8, "bf16"),
                                         (1536, 384, 1, "f32"), (520, 130, 5, "f32")])
def test_strided_queries(B, orc, d, r, H, dtype):
    """q and g as columns of [r, 3] parameter matrices (stride 3), with dq and
    dg written into columns of [r, 3] gradient matrices: same bits as
    contiguous q, g, dq, dg; the other columns are left untouched."""
    import torch
    T, n = 97, 5
    inp = synth.HostInputs(seed=23, q_std=0.5, g_kind="random")
    bank = B.Bank(T, d, r, n, dtype)
    for j in range(n):
        bank.append(inp.output(j, T, d, dtype))
    q, g = inp.query(4, r), inp.norm_weight(4, r)
    Q = torch.full((r, 3), 5.0, device="cuda")
    Gm = torch.full((r, 3), 6.0, device="cuda")
    Q[:, 1] = q
    Gm[:, 1] = g
    dQ = torch.full((r, 3), 7.0, device="cuda")
    dG = torch.full((r, 3), 8.0, device="cuda")
    rows = list(range(n))
    dout = inp.dout(4, T, d, dtype)
    out_c, lse_c = bank.route_fwd(rows, H, q, g, site_id=1)
    bank.zero_grad()
    dq_c, dg_c = bank.route_bwd(rows, H, q, g, out_c, dout, lse_c, site_id=1)
    grad_c = bank.grad.clone()
    out_s, lse_s = bank.route_fwd(rows, H, Q[:, 1], Gm[:, 1], site_id=2)
    bank.zero_grad()
    bank.route_bwd(rows, H, Q[:, 1], Gm[:, 1], out_s, dout, lse_s, dq=dQ[:, 1], dg=dG[:, 1],
                   site_id=2)
    torch.cuda.synchronize()
    assert _same_bits(out_s, out_c) and _same_bits(lse_s, lse_c)
    assert _same_bits(dQ[:, 1], dq_c) and _same_bits(dG[:, 1], dg_c)
    assert _same_bits(bank.grad, grad_c)
    assert torch.all(dQ[:, 0] == 7.0) and torch.all(dQ[:, 2] == 7.0)
    assert torch.all(dG[:, 0] == 8.0) and torch.all(dG[:, 2] == 8.0)
    # and the contiguous result is the oracle's
    srcs = [inp.host_output(j, T, d, dtype) for j in range(n)]
    qh, gh = inp.host_query(4, r), inp.host_norm_weight(4, r)
    o_r, l_r = orc.route_fwd(srcs, qh, gh, H, r=r)
    _, dq_r, dg_r = orc.route_bwd(srcs, qh, gh, inp.host_dout(4, T, d, dtype), H, r=r)
    tol = TOL[dtype]
    assert _nmax(_t64(out_c), o_r) <= tol and _nmax(_t64(lse_c), l_r) <= tol
    assert _nmax(_t64(dq_c), dq_r) <= tol and _nmax(_t64(dg_c), dg_r) <= tol


@pytest.mark.parametrize("d,r,H,dtype", [(1280, 1280, 8, "bf16"), (2048, 512, 4, "bf16"),
                                         (513, 513, 1, "f32")])
def test_changed_input_graph_replays(B, orc, d, r, H, dtype):
    """One CUDA graph holds a whole microbatch of three sites (appends with a
    block partial sum, forwards, backwards in reverse order, the gradient
    fold). It is replayed with new sources, queries and upstream gradients
    copied into its input buffers; every replay matches the oracle."""
    import torch
    T, M = 111, 3
    acc, sites = B.ar_block_schedule(M, 2)
    bank = B.Bank(T, d, r, M + 1, dtype)
    src = [torch.empty((T, d), dtype=bank.torch_dtype, device="cuda") for _ in range(M + 1)]
    qb = [torch.empty(r, device="cuda") for _ in range(M + 1)]
    gb = [torch.empty(r, device="cuda") for _ in range(M + 1)]
    db = [torch.empty((T, d), dtype=bank.torch_dtype, device="cuda") for _ in range(M + 1)]

    def fill(seed):
        inp = synth.HostInputs(seed=seed, q_std=0.5, g_kind="random")
        for t in range(M + 1):
            src[t].copy_(inp.output(t, T, d, dtype))
            qb[t].copy_(inp.query(t, r))
            gb[t].copy_(inp.norm_weight(t, r))
            db[t].copy_(inp.dout(t, T, d, dtype))
        return inp

    def step():
        bank.reset()
        outs = {}
        for t in range(M + 1):
            bank.append(src[t], acc[t])
            outs[t] = bank.route_fwd(sites[t], H, qb[t], gb[t], site_id=t)
        bank.zero_grad()
        grads = {}
        for t in reversed(range(M + 1)):
            out, lse = outs[t]
            grads[t] = bank.route_bwd(sites[t], H, qb[t], gb[t], out, db[t], lse, site_id=t)
            if t + 1 <= M and acc[t + 1] == t:
                B.ar_bank_grad_fold(bank.handle, t, t + 1)
        return outs, grads

    fill(100)
    step()                                          # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            outs, grads = step()
    torch.cuda.current_stream().wait_stream(side)
    from oracle import schedule, storage
    oplan = schedule.block_plan(M, 2)
    assert oplan["sites"] == sites
    tol = TOL[dtype]
    for seed in (101, 102, 103):
        inp = fill(seed)
        graph.replay()
        torch.cuda.synchronize()
        assert B.ar_device_error() == 0
        rows = storage.block_bank([inp.host_output(t, T, d, dtype) for t in range(M + 1)], oplan,
                                  dtype)
        dsrc = [np.zeros((T, d)) for _ in range(M + 1)]
        for t in range(M + 1):
            ss = [rows[j] for j in sites[t]]
            qh, gh = inp.host_query(t, r), inp.host_norm_weight(t, r)
            o_r, l_r = orc.route_fwd(ss, qh, gh, H, r=r)
            assert _nmax(_t64(outs[t][0]), o_r) <= tol, (seed, t)
            assert _nmax(_t64(outs[t][1]), l_r) <= tol, (seed, t)
        for t in reversed(range(M + 1)):
            ss = [rows[j] for j in sites[t]]
            qh, gh = inp.host_query(t, r), inp.host_norm_weight(t, r)
            _, dq_r, dg_r = orc.route_bwd(ss, qh, gh, inp.host_dout(t, T, d, dtype), H, r=r,
                                          dsrc=[dsrc[j] for j in sites[t]])
            assert _nmax(_t64(grads[t][0]), dq_r) <= tol, (seed, t)
            assert _nmax(_t64(grads[t][1]), dg_r) <= tol, (seed, t)
        # the adjoint of every sublayer output: its own row plus, for a block
        # partial sum, the adjoints of the later versions folded into it
        for t in range(M + 1):
            want = dsrc[t].copy()
            u = t + 1
            while u <= M and acc[u] == u - 1:
                want += dsrc[u]
                u += 1
            assert _nmax(_t64(bank.grad[t]), want) <= tol, (seed, t)

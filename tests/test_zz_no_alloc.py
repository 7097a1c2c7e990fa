"""ar_route_bwd_noalloc: the routing backward for callers that cannot allocate
device memory (its scratch lives in a fixed array inside the library).

Checked through the C ABI on two backward calls in a row, within the parity
tolerance of the fp32 tests, against the CPU oracle (every dq, dg and source
gradient) and against the regular ar_route_bwd (same bank, same inputs, a
caller-provided workspace). This file is collected last so that a
stop-at-first-failure run has already run every other test; it also passes
alone in a fresh process.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
SITES = {1: [0, 1, 2, 3, 4], 2: [0, 2, 4]}   # forward order; backward runs 2, then 1


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from depth_wise_attention_ar_gb300 import build
    build.build()
    from depth_wise_attention_ar_gb300 import binding
    return binding


def _f64(t):
    return t.detach().double().cpu().numpy()


def _nmax(x, ref):
    x = x if isinstance(x, np.ndarray) else _f64(x)
    ref = ref if isinstance(ref, np.ndarray) else _f64(ref)
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _inputs():
    """Seeded inputs of two sites over five fp32 rows (T = 777, d = 1280, H = 8)."""
    import torch
    T, d = 777, 1280
    g = torch.Generator(device="cuda")
    g.manual_seed(42)
    rows = [torch.randn((T, d), generator=g, device="cuda") / (1.0 + j) for j in range(5)]
    q = {s: 0.5 * torch.randn(d, generator=g, device="cuda") for s in SITES}
    w = {s: 1.0 + 0.1 * torch.randn(d, generator=g, device="cuda") for s in SITES}
    dout = {s: torch.randn((T, d), generator=g, device="cuda") for s in SITES}
    return rows, q, w, dout


def _run(B, noalloc: bool, inp):
    """Both sites forward, then their backwards back to back."""
    import torch
    rows, q, w, dout = inp
    T, d = rows[0].shape
    H = 8
    bank = B.Bank(T, d, d, 5, "f32")
    for j, x in enumerate(rows):
        bank.rows[j].copy_(x)
        bank.append(bank.rows[j])
    fw = {s: bank.route_fwd(lst, H, q[s], w[s], site_id=s) for s, lst in SITES.items()}
    bank.zero_grad()
    res = {}
    for s in (2, 1):  # reverse forward order
        out, lse = fw[s]
        dq = torch.empty(d, device="cuda")
        dg = torch.empty(d, device="cuda")
        if noalloc:
            B.ar_route_bwd_noalloc(bank.handle, SITES[s], H, q[s], w[s], out, dout[s], lse, dq,
                                   dg, s)
        else:
            ws = bank.workspace(H)
            B.ar_route_bwd(bank.handle, SITES[s], H, q[s], w[s], out, dout[s], lse, dq, dg, ws,
                           ws.numel() * 4, s)
        res[s] = (dq, dg)
    torch.cuda.synchronize()
    return res, bank.grad.clone()


def _oracle(inp):
    """dq, dg per site and the summed source gradients, from the CPU oracle."""
    import oracle
    rows, q, w, dout = inp
    src = [_f64(x) for x in rows]
    T, d = src[0].shape
    dsrc = [np.zeros((T, d)) for _ in src]
    res = {}
    for s in (2, 1):
        _, dq, dg = oracle.route_bwd([src[j] for j in SITES[s]], _f64(q[s]), _f64(w[s]),
                                     _f64(dout[s]), 8, dsrc=[dsrc[j] for j in SITES[s]])
        res[s] = (dq, dg)
    return res, dsrc


def test_noalloc_backward_matches_oracle_and_workspace_backward(B):
    import torch
    inp = _inputs()
    want, want_rows = _oracle(inp)
    ref, ref_grad = _run(B, noalloc=False, inp=inp)
    # two calls of the no-alloc backward in a row (each a pair of sites); the
    # second reuses the scratch the first left behind
    for _ in range(2):
        got, got_grad = _run(B, noalloc=True, inp=inp)
        assert B.ar_device_error() == 0
        assert torch.isfinite(got_grad).all()
        for s in (1, 2):
            for a, b, o in zip(got[s], ref[s], want[s]):
                assert _nmax(a, o) <= TOL_F32
                assert _nmax(a, b) <= TOL_F32
        for j in range(5):
            assert _nmax(got_grad[j], want_rows[j]) <= TOL_F32, j
        assert _nmax(got_grad, ref_grad) <= TOL_F32


def test_noalloc_rejects_workspace_beyond_its_scratch(B):
    """A bank whose backward needs more scratch than the fixed array gets
    AR_ERR_CAPACITY, launches nothing and leaves dq as it was; a bank within
    it runs. The size comes from the library itself."""
    import torch
    cap = B.ar_noalloc_scratch_bytes()
    assert cap == 8 << 20
    outcomes = {}
    for d in (8192, 512):                   # 8192 wide: ~10 MB of partial rows
        bank = B.Bank(64, d, d, 2, "bf16")
        x = torch.zeros((64, d), dtype=torch.bfloat16, device="cuda")
        bank.append(x)
        bank.append(x)
        q = torch.zeros(d, device="cuda")
        out, lse = bank.route_fwd([0, 1], 8, q, site_id=1)
        bank.zero_grad()
        need = B.ar_route_bwd_workspace(bank.handle, 8)
        dq = torch.full((d,), 3.0, device="cuda")
        if need > cap:
            with pytest.raises(B.ARError) as e:
                B.ar_route_bwd_noalloc(bank.handle, [0, 1], 8, q, None, out, out, lse, dq, None, 1)
            assert e.value.name == "AR_ERR_CAPACITY"
            torch.cuda.synchronize()
            assert torch.all(dq == 3.0)
            outcomes[d] = "refused"
        else:
            B.ar_route_bwd_noalloc(bank.handle, [0, 1], 8, q, None, out, out, lse, dq, None, 1)
            torch.cuda.synchronize()
            assert torch.all(dq == 0.0)
            outcomes[d] = "ran"
    assert outcomes == {8192: "refused", 512: "ran"}, outcomes

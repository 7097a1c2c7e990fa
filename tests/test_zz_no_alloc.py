"""ar_route_bwd_noalloc: the routing backward for callers that cannot allocate
device memory (its scratch lives in a fixed array inside the library).

Checked through the C ABI against the regular ar_route_bwd (same bank, same
inputs, a caller-provided workspace) on two backward calls in a row, within
the parity tolerance of the fp32 tests. This file is collected last so that a
stop-at-first-failure run has already run every other test; it also passes
alone in a fresh process.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5


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
    x = x.detach().double().cpu().numpy()
    ref = ref.detach().double().cpu().numpy()
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _run(B, noalloc: bool):
    """Two sites (N = 5 and N = 3) forward, then their backwards back to back."""
    import torch
    T, d, H, dtype = 777, 1280, 8, "f32"
    g = torch.Generator(device="cuda")
    g.manual_seed(42)
    bank = B.Bank(T, d, d, 5, dtype)
    for j in range(5):
        x = torch.randn((T, d), generator=g, device="cuda") / (1.0 + j)
        bank.rows[j].copy_(x)
        bank.append(bank.rows[j])
    sites = {1: [0, 1, 2, 3, 4], 2: [0, 2, 4]}
    q = {s: 0.5 * torch.randn(d, generator=g, device="cuda") for s in sites}
    w = {s: 1.0 + 0.1 * torch.randn(d, generator=g, device="cuda") for s in sites}
    dout = {s: torch.randn((T, d), generator=g, device="cuda") for s in sites}
    fw = {s: bank.route_fwd(rows, H, q[s], w[s], site_id=s) for s, rows in sites.items()}
    bank.zero_grad()
    res = {}
    for s in (2, 1):  # reverse forward order
        out, lse = fw[s]
        dq = torch.empty(d, device="cuda")
        dg = torch.empty(d, device="cuda")
        if noalloc:
            B.ar_route_bwd_noalloc(bank.handle, sites[s], H, q[s], w[s], out, dout[s], lse, dq,
                                   dg, s)
        else:
            ws = bank.workspace(H)
            B.ar_route_bwd(bank.handle, sites[s], H, q[s], w[s], out, dout[s], lse, dq, dg, ws,
                           ws.numel() * 4, s)
        res[s] = (dq, dg)
    torch.cuda.synchronize()
    return res, bank.grad.clone(), bank


def test_noalloc_backward_matches_workspace_backward(B):
    import torch
    ref, ref_grad, _ = _run(B, noalloc=False)
    got, got_grad, bank = _run(B, noalloc=True)
    assert B.ar_device_error() == 0
    for s in (1, 2):
        for a, b in zip(got[s], ref[s]):
            assert _nmax(a, b) <= TOL_F32
    assert _nmax(got_grad, ref_grad) <= TOL_F32
    # a second pair of calls reuses the shared scratch: same results again
    got2, got2_grad, _ = _run(B, noalloc=True)
    for s in (1, 2):
        for a, b in zip(got2[s], ref[s]):
            assert _nmax(a, b) <= TOL_F32
    assert _nmax(got2_grad, ref_grad) <= TOL_F32
    assert torch.isfinite(got2_grad).all()


def test_noalloc_rejects_workspace_beyond_its_scratch(B):
    """Shapes whose backward needs more scratch than the fixed array get
    AR_ERR_CAPACITY and launch nothing; shapes within it run."""
    import torch
    for d in (2048, 1280, 512):
        bank = B.Bank(64, d, d, 2, "bf16")
        x = torch.zeros((64, d), dtype=torch.bfloat16, device="cuda")
        bank.append(x)
        bank.append(x)
        q = torch.zeros(d, device="cuda")
        out, lse = bank.route_fwd([0, 1], 8, q, site_id=1)
        bank.zero_grad()
        need = B.ar_route_bwd_workspace(bank.handle, 8)
        dq = torch.full((d,), 3.0, device="cuda")
        if need > B.AR_NOALLOC_SCRATCH_BYTES:
            with pytest.raises(B.ARError) as e:
                B.ar_route_bwd_noalloc(bank.handle, [0, 1], 8, q, None, out, out, lse, dq, None, 1)
            assert e.value.name == "AR_ERR_CAPACITY"
            torch.cuda.synchronize()
            assert torch.all(dq == 3.0)
        else:
            B.ar_route_bwd_noalloc(bank.handle, [0, 1], 8, q, None, out, out, lse, dq, None, 1)
            torch.cuda.synchronize()
            assert torch.all(dq == 0.0)

"""Model-level chain through torch autograd (the routing kernels under a
stand-in model of random linear sublayers) against the float64 torch
restatement of the same model (oracle/torch_route.py): gradients of the
embedding, every sublayer weight, every query and every norm weight. Covers
the reverse-order backward, the in-place gradient accumulation across sites
and the block-sum fan-out of partial sums ("Low-Rank Attention Residuals",
Figure 11 and Appendix B.4)."""

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def AG():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from depth_wise_attention_ar_gb300 import build
    build.build()
    from depth_wise_attention_ar_gb300 import autograd
    return autograd


def _nmax(a, b):
    a = a.detach().double().cpu().numpy()
    b = b.detach().double().cpu().numpy()
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


# Every gradient is held to the fp32 bound of the rest of the parity suite
# (normalised max-abs error against the float64 chain). The stand-in model's
# sublayers run in float64 on the GPU too and round their outputs once to
# float32 at the library's boundary (the bank stores fp32), so what the
# comparison measures beyond one rounding per boundary tensor is the library's
# own arithmetic, compounded over the chain: dL/dq_t and dL/dg_t (the
# backward's dq/dg), dL/do_t (the completed adjoint of bank row t, handed back
# to autograd; for t = 0 the embedding's gradient), and the sublayer weights'
# gradients that torch forms from them.
TOL = 1e-5


@pytest.mark.parametrize("d,r,H,NB", [(512, 512, 4, None), (512, 512, 4, 3), (1024, 256, 8, 3),
                                      (1024, 256, 8, None), (1280, 1280, 8, 2)])
def test_chain_gradients_match_float64_reference(AG, d, r, H, NB):
    import torch
    from oracle import torch_route
    T, M = 300, 6
    rng = [synth.misc_normal(21, k, s, sd) for k, (s, sd) in enumerate(
        [((T, d), 1.0)] + [((d, d), 1.0 / np.sqrt(d))] * M + [((r,), 0.5)] * (M + 1)
        + [((r,), 0.1)] * (M + 1) + [((T, d), 1.0)])]
    x0, Ws = rng[0], rng[1:1 + M]
    qs = rng[1 + M:2 + 2 * M]
    gs = [1.0 + a for a in rng[2 + 2 * M:3 + 3 * M]]
    Z = rng[-1]

    def leaves(dev, dt):
        mk = lambda a: torch.tensor(a, dtype=dt, device=dev, requires_grad=True)
        return mk(x0), [mk(w) for w in Ws], [mk(q) for q in qs], [mk(g) for g in gs]

    def kept(o, store):
        o.retain_grad()
        store.append(o)
        return o

    # GPU: routing through the library, fp32 bank; sublayers in float64,
    # their outputs rounded once to float32
    x, W, q, g = leaves("cuda", torch.float32)
    router = AG.DepthRouter(T, d, H, M, r=r, NB=NB, dtype="f32", device="cuda")
    router.begin()
    os_gpu = []
    h = router.route(0, x, q[0], g[0])
    for t in range(1, M + 1):
        o = kept((torch.tanh(h.double() @ W[t - 1].double()) * 0.5).float(), os_gpu)
        h = router.route(t, o, q[t], g[t])
    (h * torch.tensor(Z, device="cuda")).sum().backward()
    torch.cuda.synchronize()

    # reference: the same model in float64 on the CPU
    xr, Wr, qr, gr = leaves("cpu", torch.float64)
    os_ref = []
    subs = [lambda hh, w=w: kept(torch.tanh(hh @ w) * 0.5, os_ref) for w in Wr]
    hr = torch_route.chain(xr, subs, qr, gr, H, r=r, NB=NB)
    (hr * torch.tensor(Z, dtype=torch.float64)).sum().backward()

    assert _nmax(h, hr) < TOL
    errs = {"do0 (embedding)": _nmax(x.grad, xr.grad)}
    for t in range(M):
        errs[f"do{t + 1}"] = _nmax(os_gpu[t].grad, os_ref[t].grad)
    for t in range(M + 1):
        errs[f"q{t}"] = _nmax(q[t].grad, qr[t].grad)
        errs[f"g{t}"] = _nmax(g[t].grad, gr[t].grad)
    for t in range(M):
        errs[f"W{t + 1}"] = _nmax(W[t].grad, Wr[t].grad)
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (bad, errs)


def test_chain_twice_reuses_the_bank(AG):
    """Two microbatches in a row through one router give the same gradients."""
    import torch
    T, d, H, M = 128, 512, 4, 4
    gen = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn((T, d), device="cuda", generator=gen, requires_grad=True)
    W = [torch.randn((d, d), device="cuda", generator=gen) / d ** 0.5 for _ in range(M)]
    q = [torch.randn(d, device="cuda", generator=gen, requires_grad=True) for _ in range(M + 1)]
    router = AG.DepthRouter(T, d, H, M, NB=2, dtype="f32", device="cuda")
    grads = []
    for _ in range(2):
        x.grad = None
        router.begin()
        h = router.route(0, x, q[0])
        for t in range(1, M + 1):
            h = router.route(t, torch.tanh(h @ W[t - 1]), q[t])
        h.square().sum().backward()
        grads.append(x.grad.clone())
    torch.cuda.synchronize()
    assert torch.equal(grads[0], grads[1])

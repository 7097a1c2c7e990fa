"""Delta form of the routing read (the MHAR page's mid-training conversion,
Sec. 3.3 and Appendix E: h = partial + alpha * routed over a learnable null
source plus block deltas, per-call stack with fresh gradients) against the
oracle, through the C ABI."""

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


@pytest.mark.parametrize("d,r,H,dtype", [(512, 512, 4, "f32"), (512, 512, 4, "bf16"),
                                         (1280, 1280, 8, "bf16"), (4096, 4096, 8, "bf16"),
                                         (4096, 4096, 8, "f32"), (1280, 256, 8, "bf16"),
                                         (1536, 384, 1, "f32"), (513, 513, 1, "f32"),
                                         (520, 130, 5, "bf16")])
@pytest.mark.parametrize("alpha", [0.0, 0.7])
def test_per_call_delta_stack(B, orc, d, r, H, dtype, alpha):
    """Every kernel family: one warp per token (512, 1280), four warps per row
    (4096), sliced keys (1280/256, 1536/384), scalar access (513, 520/130/5)."""
    import torch
    T, k = 173, 5                                   # null source + 5 block deltas
    inp = synth.HostInputs(seed=9, q_std=0.5, g_kind="random")
    bank = B.Bank(T, d, r, k + 1, dtype)
    null = inp.output(0, 1, d, dtype).reshape(d).contiguous()
    bank.append_broadcast(null)
    for j in range(1, k + 1):
        bank.append(inp.output(j, T, d, dtype))
    rows = list(range(k + 1))
    q, g = inp.query(7, r), inp.norm_weight(7, r)
    partial = inp.output(50, T, d, dtype)
    a_t = torch.tensor([alpha], device="cuda")
    out, routed, lse = bank.route_fwd_delta(rows, H, q, g, partial, a_t, site_id=1)
    bank.zero_grad()                                 # fresh gradients for this call
    dout = inp.dout(7, T, d, dtype)
    dq, dg, dal = bank.route_bwd_delta(rows, H, q, g, routed, dout, lse, a_t, site_id=1)
    dnull = bank.grad_token_sum(0)
    torch.cuda.synchronize()
    assert B.ar_device_error() == 0
    if alpha == 0.0:
        assert torch.equal(out, partial)             # closed gate: exactly the residual stream
    srcs = [np.broadcast_to(_t64(null), (T, d)).copy()] + \
           [inp.host_output(j, T, d, dtype) for j in range(1, k + 1)]
    qh, gh = inp.host_query(7, r), inp.host_norm_weight(7, r)
    h_ref, routed_ref, lse_ref = orc.route_fwd_delta(srcs, qh, gh, H, _t64(partial), alpha, r=r)
    tol = TOL[dtype]
    assert _nmax(_t64(out), h_ref) < tol
    assert _nmax(_t64(routed), routed_ref) < tol
    assert _nmax(_t64(lse), lse_ref) < tol
    ds, dq_r, dg_r, dal_r, _ = orc.route_bwd_delta(srcs, qh, gh, inp.host_dout(7, T, d, dtype), H,
                                                   alpha, r=r)
    if alpha == 0.0:
        assert torch.all(bank.grad == 0) and torch.all(dq == 0) and torch.all(dg == 0)
    else:
        for j in range(1, k + 1):
            assert _nmax(_t64(bank.grad[j]), ds[j]) < tol, j
        assert _nmax(_t64(dnull), ds[0].sum(0)) < tol
        assert _nmax(_t64(dq), dq_r) < tol and _nmax(_t64(dg), dg_r) < tol
    assert abs(dal.item() - dal_r) <= tol * max(1.0, abs(dal_r))


def test_full_size_delta_8b_sampled_tokens(B, orc):
    """The delta workload at the 8B shape (T = 8192, d = 4096, H = 8, full-width
    keys, 65 sites over the null source and 8 block deltas) in the benchmark's
    launch configuration: outputs, routed mixes, lse and source gradients of 24
    sampled tokens, dalpha and dq/dg of the last site, and the null source's
    gradient (a sum over every token)."""
    import torch
    from depth_wise_attention_ar_gb300 import workload as wl
    from oracle import schedule, storage
    cfg = wl.CONFIGS["delta_8b"]
    inputs = synth.DeviceInputs(seed=13, q_std=0.3, g_kind="random")
    mb = wl.Microbatch(cfg, cfg.H, inputs)
    mb.step()
    torch.cuda.synchronize()
    T, d, H = cfg.T, cfg.d, cfg.H
    toks = np.sort(np.random.default_rng(2).choice(T, size=24, replace=False))
    toks[0], toks[-1] = 0, T - 1
    ti = torch.as_tensor(toks, device="cuda")
    oplan = schedule.block_plan(cfg.M, cfg.NB)
    outs = [np.broadcast_to(_t64(mb.null), (len(toks), d)).copy()]
    outs += [_t64((mb.outputs[j] if j in mb.outputs else mb.bank.rows[j])[ti])
             for j in range(1, mb.n_rows)]
    rows = storage.block_bank(outs, oplan, "bf16")
    for j in range(1, mb.n_rows):
        assert np.array_equal(_t64(mb.bank.rows[j][ti]), rows[j]), j
    tol = TOL["bf16"]
    dsrc = {j: np.zeros((len(toks), d)) for j in range(mb.n_rows)}
    for s in mb.plan.run_sites:
        src = [rows[j] for j in mb.plan.sites[s]]
        a = float(mb.alpha[s].item())
        h, rt, l = orc.route_fwd_delta(src, _t64(mb.q[s]), _t64(mb.g[s]), H,
                                       _t64(mb.partial[s][ti]), a)
        assert _nmax(_t64(mb.out[s][ti]), h) < tol, s
        assert _nmax(_t64(mb.routed[s][ti]), rt) < tol, s
        assert _nmax(_t64(mb.lse[s][ti]), l) < tol, s
    for s in reversed(mb.plan.run_sites):
        src = [rows[j] for j in mb.plan.sites[s]]
        orc.route_bwd_delta(src, _t64(mb.q[s]), _t64(mb.g[s]), _t64(mb.dout[s][ti]), H,
                            float(mb.alpha[s].item()), dsrc=[dsrc[j] for j in mb.plan.sites[s]])
    for j in range(1, mb.n_rows):
        assert _nmax(_t64(mb.bank.grad[j][ti]), dsrc[j]) < tol, j
    assert _nmax(_t64(mb.bank.grad[0][ti]), dsrc[0]) < tol
    # the null source's gradient against the bank's own gradient row, summed in float64
    assert _nmax(_t64(mb.dnull), _t64(mb.bank.grad[0]).sum(0)) < 1e-5
    s = mb.plan.run_sites[-1]
    dq = np.zeros(d)
    dg = np.zeros(d)
    dal = 0.0
    for t0 in range(0, T, 1024):
        sl = slice(t0, min(T, t0 + 1024))
        src = [_t64(mb.bank.rows[j][sl]) for j in mb.plan.sites[s]]
        _, a1, b1, c1, _ = orc.route_bwd_delta(src, _t64(mb.q[s]), _t64(mb.g[s]),
                                               _t64(mb.dout[s][sl]), H, float(mb.alpha[s].item()))
        dq += a1
        dg += b1
        dal += c1
    assert _nmax(_t64(mb.dq[s]), dq) < tol and _nmax(_t64(mb.dg[s]), dg) < tol
    assert abs(mb.dalpha[s].item() - dal) <= tol * max(1.0, abs(dal))

"""Pins for the CPU oracle, against things other than the oracle itself.

* brute force: Eq. 3 of "Multi-Head Attention Residuals" (Eq. 2 at H = 1;
  the sliced keys of "Low-Rank Attention Residuals" Eq. 11) term by term in
  numpy, softmax/logsumexp from scipy;
* torch autograd (float64, CPU) on the torch restatement of the forward
  (oracle/torch_route.py), for every gradient the oracle's closed form gives
  (this also pins that restatement, which the model-chain tests use);
* central finite differences of the oracle's own forward;
* a second backward formulation (the per-head score form of the MHAR page's
  Appendix E) against the oracle's source-gradient form;
* the invariants the pages state (H=1 is single-head AttnRes, heads are
  independent slices, weights sum to one, one-hot read, zero query gives the
  mean, one source is the identity, permutation, scale invariance, gradient
  support outside the key slice, orthogonal invariance of RMSNorm).

Each pin is chosen so that a plausible slip in the oracle (dropped term, wrong
sign, wrong slice index, transposed operand) fails at least one of them.
"""

import numpy as np
import pytest
import scipy.special as sps

import synth


def _case(seed, N, T, d, H, r, qstd=0.7, gkind="random"):
    srcs = [synth.misc_normal(seed, 100 + n, (T, d), 1.0 / (1 + 0.3 * n)).astype(np.float64)
            for n in range(N)]
    q = synth.misc_normal(seed, 1, (r,), qstd).astype(np.float64)
    if gkind == "random":
        g = 1.0 + synth.misc_normal(seed, 2, (r,), 0.2).astype(np.float64)
    else:
        g = np.ones(r)
    G = synth.misc_normal(seed, 3, (T, d)).astype(np.float64)
    return srcs, q, g, G


def _per_head_sum(Y, H):
    """Sums of the last axis over each of its H equal contiguous slices."""
    return Y.reshape(*Y.shape[:-1], H, Y.shape[-1] // H).sum(-1)


def _brute_route(V, q, g, H, r, eps, full_width):
    """Brute force: normalised keys, per-head logits, softmax over sources, and
    each head's weights applied to its own value slice."""
    N, T, d = V.shape
    keys = V[..., d - r:]
    sq = V * V if full_width else keys * keys
    khat = keys / np.sqrt(sq.mean(-1, keepdims=True) + eps) * g
    logits = _per_head_sum(khat * q, H)                       # [N, T, H]
    alpha = sps.softmax(logits, axis=0)
    mixed = (np.repeat(alpha, d // H, axis=-1) * V).sum(0)    # [T, d]
    return mixed, sps.logsumexp(logits, axis=0), alpha


def _torch_route(V, q, g, H, r, eps, full_width):
    from oracle import torch_route
    return torch_route.route(list(V.unbind(0)), q, g, H, r, eps, full_width)


def _nmax(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


SHAPES = [
    # N, T, d, H, r, full_width
    (1, 5, 8, 1, 8, False),
    (3, 7, 8, 2, 8, False),
    (4, 6, 16, 4, 16, False),
    (6, 5, 32, 4, 32, False),
    (5, 4, 32, 2, 16, False),   # low-rank keys
    (6, 3, 32, 4, 8, False),    # low-rank keys, 2-wide key slices
    (5, 4, 32, 2, 16, True),    # full-width-RMS control
    (2, 9, 24, 3, 24, False),   # odd head count
]


@pytest.mark.parametrize("N,T,d,H,r,fw", SHAPES)
def test_forward_matches_brute_force(orc, N, T, d, H, r, fw):
    srcs, q, g, _ = _case(11, N, T, d, H, r)
    out, lse, alpha = orc.route_fwd(srcs, q, g, H, r=r, eps=1e-6, full_width=fw, want_alpha=True)
    ref_out, ref_lse, ref_alpha = _brute_route(np.stack(srcs), q, g, H, r, 1e-6, fw)
    assert _nmax(out, ref_out) < 1e-12
    assert _nmax(lse, ref_lse) < 1e-12
    assert _nmax(alpha, ref_alpha.transpose(1, 0, 2)) < 1e-12


@pytest.mark.parametrize("N,T,d,H,r,fw", SHAPES)
def test_backward_matches_torch_autograd(orc, N, T, d, H, r, fw):
    import torch
    srcs, q, g, G = _case(12, N, T, d, H, r)
    dsrc, dq, dg = orc.route_bwd(srcs, q, g, G, H, r=r, eps=1e-6, full_width=fw)
    V = torch.tensor(np.stack(srcs), dtype=torch.float64, requires_grad=True)
    tq = torch.tensor(q, requires_grad=True)
    tg = torch.tensor(g, requires_grad=True)
    out = _torch_route(V, tq, tg, H, r, 1e-6, fw)
    (out * torch.tensor(G)).sum().backward()
    assert _nmax(np.stack(dsrc), V.grad.numpy()) < 1e-11
    assert _nmax(dq, tq.grad.numpy()) < 1e-10
    assert _nmax(dg, tg.grad.numpy()) < 1e-10


def _score_coupling_backward(V, q, g, G, H, r, eps, full_width):
    """The backward in the per-head score form of "Multi-Head Attention
    Residuals" Appendix E (Figure 10), written out in numpy: weights recomputed
    from the log-sum-exp, the value dot products P[n,h] = <G_h, V_{n,h}> and their
    weighted sum per head, the score gradient dz = w (P - S), then the value
    path, the key path and the radial term of the key norm. The oracle instead
    follows the source-gradient form of "Low-Rank Attention Residuals" Eq. 15 /
    Eq. 21 / Eq. 22."""
    N, T, d = V.shape
    K, Kr = d // H, r // H
    tail = V[..., d - r:]
    width = d if full_width else r
    inv = 1.0 / np.sqrt(((V * V).mean(-1) if full_width else (tail * tail).mean(-1)) + eps)
    qg = q * g
    zr = _per_head_sum(tail * qg, H)
    z = inv[..., None] * zr
    w = np.exp(z - sps.logsumexp(z, axis=0)[None])
    P = _per_head_sum(V * G[None], H)
    dz = w * (P - (w * P).sum(0)[None])
    dV = np.repeat(w, K, axis=2) * G[None]                       # value path
    kz = inv[..., None] * dz
    dV[..., d - r:] += np.repeat(kz, Kr, axis=2) * qg[None, None]  # key path
    radial = (inv ** 3 / width * (dz * zr).sum(-1))[..., None]   # norm of the key
    if full_width:
        dV -= radial * V
    else:
        dV[..., d - r:] -= radial * tail
    U = (np.repeat(kz, Kr, axis=-1) * tail).sum((0, 1))
    return dV, g * U, q * U


@pytest.mark.parametrize("N,T,d,H,r,fw", SHAPES)
def test_backward_matches_score_coupling_form(orc, N, T, d, H, r, fw):
    srcs, q, g, G = _case(14, N, T, d, H, r)
    dsrc, dq, dg = orc.route_bwd(srcs, q, g, G, H, r=r, eps=1e-6, full_width=fw)
    dV, dq2, dg2 = _score_coupling_backward(np.stack(srcs), q, g, G, H, r, 1e-6, fw)
    assert _nmax(np.stack(dsrc), dV) < 1e-11
    assert _nmax(dq, dq2) < 1e-10
    assert _nmax(dg, dg2) < 1e-10


@pytest.mark.parametrize("fw,r", [(False, 16), (False, 32), (True, 16)])
def test_backward_finite_differences(orc, fw, r):
    N, T, d, H = 4, 3, 32, 4 if r == 32 else 2
    srcs, q, g, G = _case(13, N, T, d, H, r)
    dsrc, dq, dg = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=fw)

    def loss(ss, qq, gg):
        o, _ = orc.route_fwd(ss, qq, gg, H, r=r, full_width=fw)
        return float(np.sum(o * G))

    h = 1e-6
    rng = np.random.default_rng(0)
    for _ in range(12):
        n, t, c = rng.integers(N), rng.integers(T), rng.integers(d)
        sp = [s.copy() for s in srcs]
        sm = [s.copy() for s in srcs]
        sp[n][t, c] += h
        sm[n][t, c] -= h
        fd = (loss(sp, q, g) - loss(sm, q, g)) / (2 * h)
        assert abs(fd - dsrc[n][t, c]) <= 1e-6 * max(1.0, abs(fd))
    for j in rng.choice(r, size=6, replace=False):
        for which, ana in (("q", dq), ("g", dg)):
            vp, vm = (q.copy(), q.copy()) if which == "q" else (g.copy(), g.copy())
            vp[j] += h
            vm[j] -= h
            if which == "q":
                fd = (loss(srcs, vp, g) - loss(srcs, vm, g)) / (2 * h)
            else:
                fd = (loss(srcs, q, vp) - loss(srcs, q, vm)) / (2 * h)
            assert abs(fd - ana[j]) <= 1e-6 * max(1.0, abs(fd))


def test_single_head_is_attention_residuals(orc):
    """H=1 is Eq. 2 of the MHAR page: a single weight per source, shared by every coordinate."""
    N, T, d = 5, 6, 16
    srcs, q, g, _ = _case(14, N, T, d, 1, d)
    out, lse = orc.route_fwd(srcs, q, g, 1)
    V = np.stack(srcs)
    rms = np.sqrt((V * V).mean(-1) + 1e-6)                  # [N, T]
    logits = (V * (q * g)).sum(-1) / rms                    # q^T RMSNorm(s_i)
    w = np.exp(logits - logits.max(0)) / np.exp(logits - logits.max(0)).sum(0)
    assert _nmax(out, (w[..., None] * V).sum(0)) < 1e-13


@pytest.mark.parametrize("d,H,r", [(16, 4, 16), (32, 2, 16), (24, 3, 12)])
def test_heads_are_independent_single_head_reads(orc, d, H, r):
    """Head h of MHAR equals a single-head read whose query is zero outside key slice h
    (Eq. 3: a head's logits come from its key slice alone, and its weights mix its value slice alone)."""
    N, T = 4, 5
    srcs, q, g, G = _case(15, N, T, d, H, r)
    out, lse = orc.route_fwd(srcs, q, g, H, r=r)
    K, Kr = d // H, r // H
    for h in range(H):
        qm = np.zeros_like(q)
        qm[h * Kr:(h + 1) * Kr] = q[h * Kr:(h + 1) * Kr]
        o1, l1 = orc.route_fwd(srcs, qm, g, 1, r=r)
        assert _nmax(out[:, h * K:(h + 1) * K], o1[:, h * K:(h + 1) * K]) < 1e-13
        assert _nmax(lse[:, h], l1[:, 0]) < 1e-13
        Gm = np.zeros_like(G)
        Gm[:, h * K:(h + 1) * K] = G[:, h * K:(h + 1) * K]
        ds_h, dq_h, dg_h = orc.route_bwd(srcs, q, g, Gm, H, r=r)
        ds_1, dq_1, dg_1 = orc.route_bwd(srcs, qm, g, Gm, 1, r=r)
        assert _nmax(np.stack(ds_h), np.stack(ds_1)) < 1e-12
        sl = slice(h * Kr, (h + 1) * Kr)
        assert _nmax(dq_h[sl], dq_1[sl]) < 1e-12
        assert _nmax(dg_h[sl], dg_1[sl]) < 1e-12


def test_weights_sum_to_one_and_lse(orc):
    srcs, q, g, _ = _case(16, 7, 9, 32, 4, 32, qstd=2.0)
    _, lse, alpha = orc.route_fwd(srcs, q, g, 4, want_alpha=True)
    assert np.max(np.abs(alpha.sum(1) - 1.0)) < 1e-14
    assert np.all(alpha > 0)


def test_one_hot_read_when_query_scaled_up(orc):
    N, T, d, H = 5, 8, 16, 2
    srcs, q, g, G = _case(17, N, T, d, H, d, gkind="ones")
    V = np.stack(srcs)
    rms = np.sqrt((V * V).mean(-1) + 1e-6)
    z = _per_head_sum(V * q, H) / rms[..., None]
    zs = np.sort(z, axis=0)
    gap = float(np.min(zs[-1] - zs[-2]))
    assert gap > 0
    lam = 60.0 / gap
    out, _ = orc.route_fwd(srcs, lam * q, g, H)
    arg = np.argmax(z, axis=0)                               # [T, H]
    K = d // H
    exp_out = np.empty_like(out)
    for t in range(T):
        for h in range(H):
            exp_out[t, h * K:(h + 1) * K] = V[arg[t, h], t, h * K:(h + 1) * K]
    assert _nmax(out, exp_out) < 1e-12
    _, dq, dg = orc.route_bwd(srcs, lam * q, g, G, H)
    assert np.max(np.abs(dq)) < 1e-12


def test_zero_query_reads_the_mean(orc):
    N, T, d, H = 6, 5, 16, 4
    srcs, q, g, G = _case(18, N, T, d, H, d)
    out, lse = orc.route_fwd(srcs, np.zeros_like(q), g, H)
    assert _nmax(out, np.mean(np.stack(srcs), 0)) < 1e-14
    assert np.max(np.abs(lse - np.log(N))) < 1e-14
    _, dq, dg = orc.route_bwd(srcs, np.zeros_like(q), g, G, H)
    assert np.all(dg == 0.0)
    assert np.max(np.abs(dq)) > 0


def test_single_source_is_identity(orc):
    T, d, H = 7, 16, 4
    srcs, q, g, G = _case(19, 1, T, d, H, d)
    out, lse = orc.route_fwd(srcs, q, g, H)
    assert np.array_equal(out, srcs[0])
    ds, dq, dg = orc.route_bwd(srcs, q, g, G, H)
    assert np.array_equal(ds[0], G)
    assert np.all(dq == 0.0) and np.all(dg == 0.0)
    z = orc.inv_rms(srcs[0])[:, None] * _per_head_sum(srcs[0] * (q * g), H)
    assert _nmax(lse, z) < 1e-14


def test_permutation_equivariance(orc):
    N, T, d, H = 5, 6, 16, 2
    srcs, q, g, G = _case(20, N, T, d, H, d)
    perm = [3, 0, 4, 2, 1]
    o1, l1, a1 = orc.route_fwd(srcs, q, g, H, want_alpha=True)
    o2, l2, a2 = orc.route_fwd([srcs[p] for p in perm], q, g, H, want_alpha=True)
    assert _nmax(o2, o1) < 1e-14 and _nmax(l2, l1) < 1e-14
    assert _nmax(a2, a1[:, perm, :]) < 1e-14
    d1, q1, g1 = orc.route_bwd(srcs, q, g, G, H)
    d2, q2, g2 = orc.route_bwd([srcs[p] for p in perm], q, g, G, H)
    for i, p in enumerate(perm):
        assert _nmax(d2[i], d1[p]) < 1e-13
    assert _nmax(q2, q1) < 1e-12 and _nmax(g2, g1) < 1e-12


def test_source_scale_does_not_change_weights(orc):
    N, T, d, H = 4, 5, 16, 4
    srcs, q, g, _ = _case(21, N, T, d, H, d)
    _, _, a1 = orc.route_fwd(srcs, q, g, H, eps=0.0, want_alpha=True)
    s2 = list(srcs)
    s2[2] = srcs[2] * 7.5
    _, _, a2 = orc.route_fwd(s2, q, g, H, eps=0.0, want_alpha=True)
    assert _nmax(a2, a1) < 1e-13


def test_outside_key_slice_gets_only_the_direct_value_gradient(orc):
    """Cor. 2.1 of the LR-AttnRes page: with slice normalisation the gradient outside
    the key slice is alpha * dL/dout, exactly."""
    N, T, d, H, r = 5, 4, 32, 2, 8
    srcs, q, g, G = _case(22, N, T, d, H, r)
    _, _, a = orc.route_fwd(srcs, q, g, H, r=r, want_alpha=True)
    ds, _, _ = orc.route_bwd(srcs, q, g, G, H, r=r)
    K = d // H
    for n in range(N):
        direct = np.repeat(a[:, n, :], K, axis=1) * G
        assert np.array_equal(ds[n][:, :d - r], direct[:, :d - r])
        assert np.max(np.abs(ds[n][:, d - r:] - direct[:, d - r:])) > 0
    # the full-width control keeps a radial term outside the slice (Eq. 16, second line)
    ds_c, _, _ = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=True)
    _, _, ac = orc.route_fwd(srcs, q, g, H, r=r, full_width=True, want_alpha=True)
    direct_c = np.repeat(ac[:, 0, :], K, axis=1) * G
    assert np.max(np.abs(ds_c[0][:, :d - r] - direct_c[:, :d - r])) > 1e-6


def test_rms_orthogonal_invariance(orc):
    """RMSNorm(Ro) = R RMSNorm(o) for orthogonal R (LR-AttnRes Eq. 18): rotating the
    non-key coordinates leaves the weights unchanged under the full-width norm, and
    rotating the key slice together with the query leaves them unchanged under the
    slice norm (H=1). A non-Euclidean norm would break either."""
    N, T, d, r = 4, 6, 24, 8
    srcs, q, g, _ = _case(23, N, T, d, 1, r, gkind="ones")
    Qa, _ = np.linalg.qr(synth.misc_normal(1, 9, (d - r, d - r)).astype(np.float64))
    rot = [np.concatenate([s[:, :d - r] @ Qa.T, s[:, d - r:]], axis=1) for s in srcs]
    _, _, a1 = orc.route_fwd(srcs, q, g, 1, r=r, full_width=True, want_alpha=True)
    o2, _, a2 = orc.route_fwd(rot, q, g, 1, r=r, full_width=True, want_alpha=True)
    assert _nmax(a2, a1) < 1e-13
    Qb, _ = np.linalg.qr(synth.misc_normal(1, 10, (r, r)).astype(np.float64))
    rot_k = [np.concatenate([s[:, :d - r], s[:, d - r:] @ Qb.T], axis=1) for s in srcs]
    _, _, b1 = orc.route_fwd(srcs, q, g, 1, r=r, want_alpha=True)
    _, _, b2 = orc.route_fwd(rot_k, Qb @ q, g, 1, r=r, want_alpha=True)
    assert _nmax(b2, b1) < 1e-13


def test_low_rank_with_full_key_width_is_plain_routing(orc):
    """r = d reduces LR-AttnRes to AttnRes (LR page, Sec. 3.3); the slice norm and the
    full-width norm then coincide."""
    srcs, q, g, G = _case(24, 4, 5, 16, 2, 16)
    o1, l1 = orc.route_fwd(srcs, q, g, 2, r=16, full_width=False)
    o2, l2 = orc.route_fwd(srcs, q, g, 2, r=16, full_width=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_inv_rms_definition(orc):
    x = np.array([[3.0, 4.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0]])
    inv = orc.inv_rms(x, r=4, eps=0.0)
    assert np.allclose(inv, [1.0 / np.sqrt(25.0 / 4.0), 1.0], rtol=0, atol=1e-15)
    inv_tail = orc.inv_rms(x, r=2, eps=0.0)
    assert inv_tail[1] == 1.0 and np.isinf(inv_tail[0])


@pytest.mark.parametrize("NB", [None, 2, 3])
def test_torch_chain_matches_schedule_and_c_oracle(orc, NB):
    """The float64 model chain (oracle/torch_route.chain) against the block
    schedule, the storage of partial sums and the C oracle, read by read."""
    import torch
    from oracle import schedule, torch_route
    T, d, H, M = 5, 16, 2, 6
    Ws = [synth.misc_normal(31, t, (d, d), 0.3).astype(np.float64) for t in range(M)]
    qs = [synth.misc_normal(32, t, (d,), 0.8).astype(np.float64) for t in range(M + 1)]
    x = synth.misc_normal(33, 0, (T, d)).astype(np.float64)
    subs = [lambda hh, w=torch.tensor(w): torch.tanh(hh @ w) for w in Ws]
    h_chain = torch_route.chain(torch.tensor(x), subs, [torch.tensor(q) for q in qs],
                                [None] * (M + 1), H, NB=NB).numpy()
    plan = schedule.block_plan(M, NB)
    outs = [x]
    h, _ = orc.route_fwd([x], qs[0], None, H)
    for t in range(1, M + 1):
        outs.append(np.tanh(h @ Ws[t - 1]))
        rows = _exact_block_rows(outs, plan, t)     # block sums without rounding
        h, _ = orc.route_fwd([rows[j] for j in plan["sites"][t]], qs[t], None, H)
    assert np.max(np.abs(h - h_chain)) < 1e-12


def _exact_block_rows(outs, plan, t):
    rows = []
    for op in plan["row_ops"][:t + 1]:
        if op[0] in ("emb", "copy"):
            rows.append(outs[0] if op[0] == "emb" else outs[op[1]])
        else:
            rows.append(rows[op[1]] + outs[op[2]])
    return rows


def test_delta_form_closed_gate_is_identity(orc):
    """alpha = 0: the delta form returns the residual stream exactly (the
    identity-preserving conversion of the MHAR page, Sec. 3.3); its dalpha is
    <dout, routed> summed, the source gradients vanish and dpartial = dout."""
    srcs, q, g, G = _case(40, 4, 6, 16, 4, 16)
    P = synth.misc_normal(40, 99, (6, 16)).astype(np.float64)
    h, routed, lse = orc.route_fwd_delta(srcs, q, g, 4, P, 0.0)
    assert np.array_equal(h, P)
    ds, dq, dg, dalpha, dpart = orc.route_bwd_delta(srcs, q, g, G, 4, 0.0)
    assert all(np.all(x == 0) for x in ds) and np.all(dq == 0) and np.all(dg == 0)
    assert abs(dalpha - float(np.sum(G * routed))) == 0.0 and np.array_equal(dpart, G)


def test_delta_form_matches_autograd_and_finite_differences(orc):
    import torch
    from oracle import torch_route
    srcs, q, g, G = _case(41, 5, 7, 32, 4, 16)
    P = synth.misc_normal(41, 98, (7, 32)).astype(np.float64)
    alpha = 0.37
    ds, dq, dg, dalpha, dpart = orc.route_bwd_delta(srcs, q, g, G, 4, alpha, r=16)
    V = [torch.tensor(s_, requires_grad=True) for s_ in srcs]
    tq, tg = torch.tensor(q, requires_grad=True), torch.tensor(g, requires_grad=True)
    ta, tp = torch.tensor(alpha, dtype=torch.float64, requires_grad=True), torch.tensor(P, requires_grad=True)
    h = tp + ta * torch_route.route(V, tq, tg, 4, r=16)
    (h * torch.tensor(G)).sum().backward()
    for n in range(5):
        assert _nmax(ds[n], V[n].grad.numpy()) < 1e-11
    assert _nmax(dq, tq.grad.numpy()) < 1e-10 and _nmax(dg, tg.grad.numpy()) < 1e-10
    assert abs(dalpha - ta.grad.item()) < 1e-10 * max(1.0, abs(dalpha))
    assert np.array_equal(dpart, G)
    eps = 1e-6
    hp, _, _ = orc.route_fwd_delta(srcs, q, g, 4, P, alpha + eps, r=16)
    hm, _, _ = orc.route_fwd_delta(srcs, q, g, 4, P, alpha - eps, r=16)
    fd = float(np.sum((hp - hm) * G)) / (2 * eps)
    assert abs(fd - dalpha) <= 1e-6 * max(1.0, abs(fd))


def test_lse_merge_of_disjoint_source_sets(orc):
    """The read over A u B is the log-sum-exp merge of the reads over A and B,
    per head (the online-softmax update two-phase inference relies on)."""
    srcs, q, g, _ = _case(42, 7, 5, 16, 4, 16, qstd=1.5)
    oa, la = orc.route_fwd(srcs[:4], q, g, 4)
    ob, lb = orc.route_fwd(srcs[4:], q, g, 4)
    o, l = orc.route_fwd(srcs, q, g, 4)
    lse = np.logaddexp(la, lb)
    K = 4
    wa = np.repeat(np.exp(la - lse), K, axis=1)
    wb = np.repeat(np.exp(lb - lse), K, axis=1)
    assert _nmax(lse, l) < 1e-14
    assert _nmax(wa * oa + wb * ob, o) < 1e-13


@pytest.mark.parametrize("N,T,d,H,r,fw", [(5, 17, 64, 4, 64, False), (9, 11, 96, 2, 32, False),
                                          (4, 13, 64, 8, 32, True), (1, 7, 32, 1, 32, False)])
def test_float32_build_agrees_with_float64(orc, N, T, d, H, r, fw):
    """The float32 build (the same C source compiled with -DORC_FLOAT, which
    the benchmark times as the CPU baseline) against the float64 reference
    pinned above: forward, lse, every source gradient, dq and dg within the
    fp32 bound of the parity suite. The float32 library really computes in
    float32 (its type size is checked on load), so its results differ from
    the float64 ones, but only by rounding."""
    srcs, q, g, G = _case(13, N, T, d, H, r)
    srcs32 = [s.astype(np.float32) for s in srcs]
    out64, lse64 = orc.route_fwd(srcs32, q.astype(np.float32), g.astype(np.float32), H, r=r,
                                 full_width=fw)
    out32, lse32 = orc.route_fwd(srcs32, q, g, H, r=r, full_width=fw, precision="f32")
    assert out32.dtype == np.float32 and lse32.dtype == np.float32

    def nmax(x, ref):
        return float(np.max(np.abs(x.astype(np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))

    assert nmax(out32, out64) < 1e-5 and nmax(lse32, lse64) < 1e-5
    assert 0 < nmax(out32, out64) or N == 1        # rounding differs: a real float32 build
    ds64, dq64, dg64 = orc.route_bwd(srcs32, q.astype(np.float32), g.astype(np.float32),
                                     G.astype(np.float32), H, r=r, full_width=fw)
    ds32, dq32, dg32 = orc.route_bwd(srcs32, q, g, G, H, r=r, full_width=fw, precision="f32")
    for a, b in zip(ds32, ds64):
        assert nmax(a, b) < 1e-5
    if N > 1:
        assert nmax(dq32, dq64) < 1e-5 and nmax(dg32, dg64) < 1e-5
    else:
        assert np.all(dq32 == 0) and np.all(dg32 == 0)
    inv32 = orc.inv_rms(srcs32[0], r=r, full_width=fw, precision="f32")
    assert nmax(inv32, orc.inv_rms(srcs32[0], r=r, full_width=fw)) < 1e-6


@pytest.mark.parametrize("N,T,d,H,r,fw", [(5, 9, 64, 4, 64, False), (4, 7, 96, 1, 32, False),
                                          (3, 5, 64, 8, 32, True)])
def test_backward_coupling_from_a_given_forward_output(orc, N, T, d, H, r, fw):
    """route_bwd(fwd_out=...): the forward output enters the backward only
    through its per-head dot with dL/dout (the coupling of the sources in the
    routing feedback, "Multi-Head Attention Residuals", Appendix E). So:
    the oracle's own forward output gives the recomputing backward's result;
    an output changed orthogonally to dL/dout within every head gives the same
    result again; a change along dL/dout changes the result linearly (twice
    the change, twice the difference) and not at all the direct value term
    outside the key slice."""
    srcs, q, g, G = _case(17, N, T, d, H, r)
    out, _ = orc.route_fwd(srcs, q, g, H, r=r, full_width=fw)
    ref = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=fw)
    same = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=fw, fwd_out=out)
    for a, b in zip(ref[0] + list(ref[1:]), same[0] + list(same[1:])):
        assert _nmax(b, a) < 1e-12
    K = d // H
    rng = np.random.default_rng(5)
    X = rng.normal(size=(T, d))
    for t in range(T):                         # X_[h] orthogonal to G_[h] in every head
        for h in range(H):
            sl = slice(h * K, (h + 1) * K)
            gh = G[t, sl]
            X[t, sl] -= gh * np.dot(gh, X[t, sl]) / np.dot(gh, gh)
    orth = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=fw, fwd_out=out + 0.3 * X)
    for a, b in zip(ref[0] + list(ref[1:]), orth[0] + list(orth[1:])):
        assert _nmax(b, a) < 1e-10
    d1 = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=fw, fwd_out=out + 1e-3 * G)
    d2 = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=fw, fwd_out=out + 2e-3 * G)
    for n in range(N):
        e1, e2 = d1[0][n] - ref[0][n], d2[0][n] - ref[0][n]
        assert np.max(np.abs(e1)) > 0 or N == 1
        assert np.max(np.abs(e2 - 2 * e1)) <= 1e-8 * max(np.max(np.abs(e2)), 1e-30)
        if not fw and r < d:                   # only key / RMS coordinates feel the coupling
            assert np.max(np.abs(e1[:, : d - r])) == 0
    # the float32 build takes the same argument
    f32 = orc.route_bwd(srcs, q, g, G, H, r=r, full_width=fw, fwd_out=out + 1e-3 * G,
                        precision="f32")
    for a, b in zip(d1[0], f32[0]):
        assert _nmax(b.astype(np.float64), a) < 1e-5

"""Depth routing inside a torch autograd graph, through the C ABI.

``DepthRouter`` serves one model: at every read site it appends the newest
sublayer output to the bank and routes, as a ``torch.autograd.Function``
("Multi-Head Attention Residuals", Figure 3 and Appendix E; "Low-Rank
Attention Residuals", Figure 11):

    router.begin()
    h = router.route(0, x, q[0], g[0])               # x: token embedding
    for t in 1..M:
        o = sublayer_t(h)
        h = router.route(t, o, q[t], g[t])           # reads blocks + partial
    loss(h).backward()

Backward of site t (autograd runs them in strictly reverse order, which the
library checks): ``ar_route_bwd`` adds dL/ds for every row the site read into
the shared fp32 gradient rows (store on a row's first touch, then in place),
and returns dL/dq, dL/dg. Row t is first read at site t, so by then every later
site has added its share; with block routing, row t+1 = row t + o_{t+1} also
hands its whole adjoint down (``ar_bank_grad_fold``, the block-sum fan-out).
The completed adjoint of row t is dL/do_t, handed back to autograd — the only
source gradient autograd sees; the others travel through the bank.

All computation runs in the library's kernels; this module only sequences the
calls and hands tensors to autograd (a dtype cast of the returned gradient
when the bank stores bf16).
"""

from __future__ import annotations

import torch

from . import binding as B

__all__ = ["DepthRouter"]


class DepthRouter:
    def __init__(self, T: int, d: int, H: int, M: int, r: int | None = None,
                 NB: int | None = None, dtype: str = "bf16", norm: str = "key",
                 eps: float = 1e-6, device=None):
        self.T, self.d, self.H, self.M = T, d, H, M
        self.r = d if r is None else r
        self.acc_from, self.sites = B.ar_block_schedule(M, NB)
        self.bank = B.Bank(T, d, self.r, M + 1, dtype, norm=norm, eps=eps, device=device)
        self._bwd_started = False

    def begin(self):
        """Start a microbatch: forget rows and routing records."""
        self.bank.reset()
        self._bwd_started = False

    def route(self, t: int, o_t: torch.Tensor, q: torch.Tensor, g: torch.Tensor | None = None):
        """Append o_t as bank row t and return the read of site t (the input of
        sublayer t+1, or of the head after the last sublayer)."""
        if self.bank.count != t:
            raise RuntimeError(f"site {t} routed out of order (bank holds {self.bank.count} rows)")
        return _RouteFn.apply(self, t, o_t, q, g)


class _RouteFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, router: DepthRouter, t: int, o_t, q, g):
        bank = router.bank
        src = o_t.detach().contiguous()
        bank.append(src, router.acc_from[t])
        out, lse = bank.route_fwd(router.sites[t], router.H, q.detach().contiguous(),
                                  None if g is None else g.detach().contiguous(), site_id=t)
        ctx.router, ctx.t, ctx.has_g = router, t, g is not None
        ctx.o_dtype = o_t.dtype
        ctx.save_for_backward(q, g if g is not None else q, out, lse)
        return out

    @staticmethod
    def backward(ctx, dout):
        router, t = ctx.router, ctx.t
        bank = router.bank
        q, g, out, lse = ctx.saved_tensors
        g = g if ctx.has_g else None
        if not router._bwd_started:
            bank.zero_grad()
            router._bwd_started = True
        dq, dg = bank.route_bwd(router.sites[t], router.H, q.detach().contiguous(),
                                None if g is None else g.detach().contiguous(), out,
                                dout.to(bank.torch_dtype).contiguous(), lse, site_id=t)
        if t + 1 <= router.M and router.acc_from[t + 1] == t:
            B.ar_bank_grad_fold(bank.handle, t, t + 1)
        # a copy: the bank's rows are reused by the next microbatch, and a leaf
        # (the embedding) would otherwise keep a view of them as its .grad
        d_o = bank.grad[t].to(ctx.o_dtype, copy=True)
        return None, None, d_o, dq, dg

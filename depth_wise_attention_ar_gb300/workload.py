"""Microbatch driver: the whole routing path of one microbatch through the C ABI.

A microbatch is what one training step of a model with depth routing asks of
this library ("Multi-Head Attention Residuals", Figure 3 and Appendix E;
"Low-Rank Attention Residuals", Figure 11):

1. forward, in model order: append each new source row (its inverse RMS is
   computed once here) and run the forward of every routing site;
2. backward, in reverse order: run the backward of every site, accumulating
   dL/ds into the shared fp32 gradient rows and producing dL/dq, dL/dg.

Bank layout: row 0 holds the embedding, row t the state after sublayer t —
the sublayer output itself (full routing) or the block partial sum
(block routing). Rows that are plain sublayer outputs are written in place by
their producer (here: filled before the step) and appended without a copy;
block partial sums are appended as row p + o_t from a separate output buffer.

The schedule comes from the library's own bookkeeping (``ar_block_schedule``);
full routing is the schedule with one block per sublayer.
"""

from __future__ import annotations

from dataclasses import dataclass, field


__all__ = ["Config", "CONFIGS", "Plan", "make_plan", "Microbatch", "model_bytes"]


@dataclass(frozen=True)
class Config:
    name: str
    T: int                      # tokens per microbatch (batch x sequence)
    d: int                      # width
    H: int                      # routing heads
    r: int                      # key width (r = d: full keys)
    dtype: str                  # "bf16" | "f32"
    M: int                      # residual-writing sublayers (2L)
    NB: int | None = None       # blocks (None: full routing)
    sites: tuple | None = None  # restrict to these site indices (None: all)
    q_std: float = 0.02
    norm: str = "key"           # RMS over the key coordinates, or "full" width
    delta: bool = False         # delta form: row 0 is a learnable null source, every
                                # site returns partial + alpha * routed
    note: str = ""


CONFIGS = {
    "tiny": Config("tiny", T=256, d=512, H=4, r=512, dtype="f32", M=4, sites=(4,),
                   note="one MHAR site over N=5 sources, fp32"),
    "100M": Config("100M", T=8 * 2048, d=512, H=4, r=512, dtype="bf16", M=24,
                   note="d=512, L=12: 25 sites, site i reads the first i sources"),
    "350M": Config("350M", T=16 * 1024, d=1024, H=8, r=1024, dtype="bf16", M=48,
                   note="d=1024, L=24: 49 sites"),
    "1B": Config("1B", T=16 * 1024, d=1280, H=8, r=1280, dtype="bf16", M=72,
                 note="d=1280, L=36: 73 sites"),
    "lr_block": Config("lr_block", T=8192, d=4096, H=8, r=1024, dtype="bf16", M=64, NB=8,
                       note="32 layers in 8 blocks, keys = last 1024 coordinates"),
    "lr_page_1b": Config("lr_page_1b", T=2 * 2048, d=1536, H=1, r=384, dtype="bf16", M=48, NB=8,
                         note="the LR page's 1B model: 24 layers, 8 blocks, r = d/4, one head"),
    "lr_page_4b": Config("lr_page_4b", T=2 * 2048, d=2560, H=1, r=640, dtype="bf16", M=88, NB=8,
                         note="the LR page's 4B model: 44 layers, 8 blocks, r = d/4, one head"),
    "delta_8b": Config("delta_8b", T=2 * 4096, d=4096, H=8, r=4096, dtype="bf16", M=64, NB=8,
                       delta=True,
                       note="delta form of the 8B mid-training model: null source + 8 block "
                            "deltas (at most 9 sources), H=8, full-width keys"),
}


@dataclass
class Plan:
    acc_from: list            # per bank row: -1 (stored as is) or the row it accumulates onto
    sites: list               # per site: row list
    run_sites: list           # site indices that run

    @property
    def rows(self) -> int:
        return len(self.acc_from)


def make_plan(cfg: Config) -> Plan:
    from . import binding as B
    acc, sites = B.ar_block_schedule(cfg.M, cfg.NB)
    run = list(cfg.sites) if cfg.sites is not None else list(range(len(sites)))
    return Plan(acc_from=acc, sites=sites, run_sites=run)


def model_bytes(cfg: Config, plan: Plan, H: int | None = None) -> dict:
    """Algorithmic bytes of one microbatch (what the method must move).

    forward site : T (N b d + 4 N + b d + 4 H)   (rows, inverse RMS, out, lse)
    backward site: T (b d + 4 H + 4 N + N b d + N d (8, or 4 on a row's first
                   touch))                       (dout, lse, inverse RMS, rows
                                                  once, gradient rows)
    The backward kernel also reads the forward output once per token (its
    softmax coupling term); that T b d is not part of the method's bytes and
    is not counted.
    append       : T (b r + 4) for a row written in place by its producer
                   (key read for the inverse RMS), T (3 b d + 4) for a partial
                   sum (two reads, one write).
    delta form   : each forward also reads the residual stream and writes the
                   routed mix (2 T b d); the null source is a broadcast fill
                   (T (b d + 4)) and its gradient a token sum (T d 4).
    """
    H = cfg.H if H is None else H
    b = 2 if cfg.dtype == "bf16" else 4
    T, d, r = cfg.T, cfg.d, cfg.r
    fwd = bwd = app = 0
    touched = set()
    needed = sorted({row for s in plan.run_sites for row in plan.sites[s]})
    for row in needed:
        if row == 0 and cfg.delta:
            app += T * (b * d + 4) + T * d * 4     # broadcast fill; its gradient's token sum
        else:
            app += T * (3 * b * d + 4) if plan.acc_from[row] >= 0 else T * (b * r + 4)
    for s in plan.run_sites:
        N = len(plan.sites[s])
        fwd += T * (N * b * d + 4 * N + b * d + 4 * H)
        if cfg.delta:
            fwd += 2 * T * b * d                    # partial read, routed mix written
    for s in reversed(plan.run_sites):
        rows = plan.sites[s]
        N = len(rows)
        g = sum(4 * d if row in touched else 0 for row in rows) + 4 * d * N
        touched.update(rows)
        bwd += T * (b * d + 4 * H + 4 * N + N * b * d) + T * g
    return {"fwd": fwd, "bwd": bwd, "append": app, "total": fwd + bwd + app}


@dataclass
class Microbatch:
    """Device buffers and launch sequence of one microbatch of a config."""

    cfg: Config
    H: int
    inputs: object            # provides output(j,T,d,dtype), query(site,r),
                              # norm_weight(site,r) (None = ones), dout(site,T,d,dtype)
    device: str = "cuda"
    plan: Plan = field(init=False)

    def __post_init__(self):
        import torch

        from . import binding as B
        cfg, dev, src = self.cfg, torch.device(self.device), self.inputs
        self.plan = make_plan(cfg)
        needed = sorted({row for s in self.plan.run_sites for row in self.plan.sites[s]})
        self.n_rows = max(needed) + 1
        self.bank = B.Bank(cfg.T, cfg.d, cfg.r, self.n_rows, cfg.dtype, norm=cfg.norm, eps=1e-6,
                           device=dev)
        tdt = self.bank.torch_dtype
        # sublayer outputs: written in place into their bank rows, or kept in
        # separate buffers when the row is a block partial sum
        self.outputs = {}
        for j in range(self.n_rows):
            if j == 0 and cfg.delta:
                # learnable null source: one vector, broadcast over the tokens
                self.null = src.output(0, 1, cfg.d, cfg.dtype).reshape(cfg.d).contiguous()
                continue
            x = src.output(j, cfg.T, cfg.d, cfg.dtype)
            if self.plan.acc_from[j] >= 0:
                self.outputs[j] = x
            else:
                self.bank.rows[j].copy_(x)
            del x
        run = self.plan.run_sites
        # per-site queries, norm weights (and gates) live in one buffer, and
        # their gradients in another, so that a host pipeline moves each set
        # with one copy
        q = {s: src.query(s, cfg.r) for s in run}
        g = {s: src.norm_weight(s, cfg.r) for s in run}
        alpha = {s: src.query(2000 + s, 1) for s in run} if cfg.delta else {}
        parts = [*q.values(), *(x for x in g.values() if x is not None), *alpha.values()]
        self.small_in = torch.cat([x.reshape(-1).float() for x in parts])
        off = 0

        def view(x):
            nonlocal off
            v = self.small_in[off:off + x.numel()].view(x.shape)
            off += x.numel()
            return v

        self.q = {s: view(q[s]) for s in run}
        self.g = {s: view(g[s]) if g[s] is not None else None for s in run}
        if cfg.delta:
            self.alpha = {s: view(alpha[s]) for s in run}
        del q, g, alpha, parts
        self.dout = {s: src.dout(s, cfg.T, cfg.d, cfg.dtype) for s in self.plan.run_sites}
        self.out = {s: torch.empty((cfg.T, cfg.d), dtype=tdt, device=dev)
                    for s in self.plan.run_sites}
        self.lse = {s: torch.empty((cfg.T, self.H), dtype=torch.float32, device=dev)
                    for s in self.plan.run_sites}
        ns = len(run)
        n_out = 2 * ns * cfg.r + ((ns + cfg.d) if cfg.delta else 0)
        self.small_out = torch.empty(n_out, device=dev)
        so = self.small_out
        self.dq = {s: so[i * cfg.r:(i + 1) * cfg.r] for i, s in enumerate(run)}
        self.dg = {s: so[(ns + i) * cfg.r:(ns + i + 1) * cfg.r] for i, s in enumerate(run)}
        self.ws = self.bank.workspace(self.H)
        if cfg.delta:
            self.partial = {s: src.output(1000 + s, cfg.T, cfg.d, cfg.dtype)
                            for s in self.plan.run_sites}
            self.routed = {s: torch.empty((cfg.T, cfg.d), dtype=tdt, device=dev)
                           for s in self.plan.run_sites}
            base = 2 * ns * cfg.r
            self.dalpha = {s: so[base + i:base + i + 1] for i, s in enumerate(run)}
            self.dnull = so[base + ns:base + ns + cfg.d]

    def forward(self, stream=None, on_site=None):
        bank, plan = self.bank, self.plan
        bank.reset()
        appended = 0
        run = set(plan.run_sites)
        last = max(plan.run_sites)
        delta = self.cfg.delta
        self.fused_appends = 0
        for t in range(last + 1):
            if on_site:
                on_site("fwd_begin", t)
            if t < self.n_rows and not delta and t in run:
                # append and read in one call: fused into one launch when the
                # row sits in its slot and the site runs on the one-warp kernels
                src = self.outputs.get(t, bank.rows[t])
                _, _, _, fused = bank.route_fwd_append(src, plan.acc_from[t], plan.sites[t], self.H,
                                                       self.q[t], self.g[t], self.out[t],
                                                       self.lse[t], site_id=t, stream=stream)
                self.fused_appends += int(fused)
                appended += 1
                if on_site:
                    on_site("fwd", t)
                continue
            if t < self.n_rows:
                if t == 0 and delta:
                    bank.append_broadcast(self.null, stream)
                else:
                    src = self.outputs.get(t, bank.rows[t])
                    bank.append(src, plan.acc_from[t], stream)
                appended += 1
            if t in run:
                if delta:
                    bank.route_fwd_delta(plan.sites[t], self.H, self.q[t], self.g[t],
                                         self.partial[t], self.alpha[t], self.out[t],
                                         self.routed[t], self.lse[t], site_id=t, stream=stream)
                else:
                    bank.route_fwd(plan.sites[t], self.H, self.q[t], self.g[t], self.out[t],
                                   self.lse[t], site_id=t, stream=stream)
                if on_site:
                    on_site("fwd", t)
        return appended

    def backward(self, stream=None, on_site=None, exact=False):
        """Every site's backward in reverse; exact=True sums each site's coupling
        term over its sources first (ar_route_bwd_exact; plain form only)."""
        bank, plan = self.bank, self.plan
        if exact and self.cfg.delta:
            raise ValueError("exact coupling is wired for the plain form here")
        bank.zero_grad()
        for t in reversed(plan.run_sites):
            if on_site:
                on_site("bwd_begin", t)
            dg = self.dg[t] if self.g[t] is not None else None
            if self.cfg.delta:
                bank.route_bwd_delta(plan.sites[t], self.H, self.q[t], self.g[t], self.routed[t],
                                     self.dout[t], self.lse[t], self.alpha[t], self.dq[t], dg,
                                     self.dalpha[t], site_id=t, stream=stream, ws=self.ws)
            else:
                bank.route_bwd(plan.sites[t], self.H, self.q[t], self.g[t], self.out[t],
                               self.dout[t], self.lse[t], self.dq[t], dg, site_id=t,
                               stream=stream, ws=self.ws, exact=exact)
            if on_site:
                on_site("bwd_end", t)
        if self.cfg.delta:
            bank.grad_token_sum(0, self.dnull, stream)   # the null source's gradient

    def step(self, stream=None):
        self.forward(stream)
        self.backward(stream)

    def kernel_launches(self) -> int:
        """Kernels one step launches: appends (those fused into their site's forward
        excepted, as counted by the last forward), forwards, backward + reduce per site."""
        fused = getattr(self, "fused_appends", 0)
        return (self.n_rows - fused + 3 * len(self.plan.run_sites) +
                (1 if self.cfg.delta else 0))

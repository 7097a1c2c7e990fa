"""Plain PyTorch (float64, CPU) restatement of one routing site and of a whole
routed model chain — test infrastructure only.

``route`` restates one routing read of "Multi-Head Attention Residuals"
(Eq. 3; Eq. 2 at H = 1) with the sliced keys of "Low-Rank Attention
Residuals" (Eq. 11): normalised keys, one logit per (source, head), softmax
over the sources, each head's weights on its own value slice. Being plain
torch ops, it is differentiable by autograd, so a routed model chain built
from it gives reference gradients for every parameter.

Pinned by tests/test_oracle_pins.py against the C oracle (forward values and,
through autograd, the closed-form gradients).
"""

from __future__ import annotations

import torch

__all__ = ["route", "chain"]


def route(sources, q, g, H: int, r: int | None = None, eps: float = 1e-6,
          full_width: bool = False):
    """sources: list of N tensors [T, d]; q, g: [r] (g None = ones)."""
    V = torch.stack(list(sources))
    N, T, d = V.shape
    r = d if r is None else r
    keys = V[..., d - r:]
    sq = V * V if full_width else keys * keys
    khat = keys * torch.rsqrt(sq.mean(-1, keepdim=True) + eps)
    if g is not None:
        khat = khat * g
    logits = (khat * q).reshape(N, T, H, r // H).sum(-1)     # one per (source, head)
    alpha = torch.softmax(logits, dim=0)                     # over the sources
    return (alpha.repeat_interleave(d // H, dim=-1) * V).sum(0)


def chain(x, sublayers, queries, norm_weights, H: int, r: int | None = None, NB: int | None = None,
          eps: float = 1e-6, full_width: bool = False):
    """A routed model (LR-AttnRes Figure 11 with MHAR heads): h = x; after each
    sublayer, route over the embedding, the completed block sums and the
    current partial sum. ``NB=None`` keeps every output as its own source
    (full routing, MHAR Figure 3). ``queries``/``norm_weights`` hold one entry
    per read (len(sublayers) + 1, the first for the read that feeds sublayer
    1). Returns the final read."""
    import bisect

    from .schedule import block_ends
    ends = block_ends(len(sublayers), NB)
    sums = []    # sums[k]: block k's outputs added up so far
    h = route([x], queries[0], norm_weights[0], H, r, eps, full_width)
    for t, f in enumerate(sublayers, start=1):
        k = bisect.bisect_left(ends, t)    # the block holding sublayer t
        o = f(h)
        if k == len(sums):
            sums.append(o)                 # first sublayer of block k
        else:
            sums[k] = sums[k] + o
        # the embedding, the finished blocks and block k up to sublayer t
        h = route([x] + sums, queries[t], norm_weights[t], H, r, eps, full_width)
    return h

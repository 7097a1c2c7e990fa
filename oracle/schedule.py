"""Source schedules: which bank rows each routing site reads (oracle side).

Full routing ("Multi-Head Attention Residuals", Sec. 2.2 and Figure 3;
"Low-Rank Attention Residuals", Eq. 4): the sources are the token embedding
plus every sublayer output, N = 2L+1 in all; routing site i (1-based) reads
the first i sources, since each sublayer's output joins the bank unchanged.

Block routing ("Low-Rank Attention Residuals", Eq. 5-6 and Figure 11): the
M = 2L sublayers fall into NB consecutive blocks, block k ending at sublayer
ceil(M*(k+1)/NB). A block's source is the sum of its sublayers' outputs. The
read after sublayer t, which lies in block k, sees the embedding and the sums
of blocks 0..k, block k's sum taken only up to sublayer t (the partial sum;
when t ends the block it is the whole block sum). So the source list grows
by one entry at each block start and otherwise has its last entry replaced.

Bank layout used by both sides of the parity checks: row 0 holds the
embedding; in full routing row j holds sublayer output j; in block routing
row t (1..M) holds the partial sum right after sublayer t, kept as an
immutable version so that the backward of every site sees the value its
forward read (a completed block is the last version of its block).
"""

from __future__ import annotations

import bisect

__all__ = ["full_sites", "block_ends", "block_plan"]


def full_sites(num_sources: int) -> list[list[int]]:
    """Row lists of full routing: site i (i = 1..num_sources) reads rows 0..i-1."""
    if num_sources < 1:
        raise ValueError("need at least one source")
    return [list(range(i)) for i in range(1, num_sources + 1)]


def block_ends(M: int, NB: int | None = None) -> list[int]:
    """Block end sublayers {ceil(M*j/NB) : j = 1..NB}; NB=None means NB = M."""
    if M < 1:
        raise ValueError("need at least one sublayer")
    nb = M if NB is None else min(NB, M)
    if nb < 1:
        raise ValueError("need at least one block")
    return sorted({(M * j + nb - 1) // nb for j in range(1, nb + 1)})


def block_plan(M: int, NB: int | None = None) -> dict:
    """Bank rows and per-site row lists of block routing over M sublayers.

    Returns a dict with
      ``ends``    : sorted block-end sublayers,
      ``row_ops`` : ``row_ops[0] = ("emb",)``; for t = 1..M either
                    ``("copy", t)`` (row t = o_t, the first write of a block)
                    or ``("acc", p, t)`` (row t = row p + o_t),
      ``sites``   : ``sites[0] = [0]`` (the read that feeds sublayer 1) and
                    ``sites[t]`` = completed block rows + [current partial row]
                    for the read after sublayer t.
    """
    ends = block_ends(M, NB)
    row_ops: list[tuple] = [("emb",)]
    sites = [[0]]
    for t in range(1, M + 1):
        k = bisect.bisect_left(ends, t)            # the block holding sublayer t
        start = ends[k - 1] + 1 if k else 1        # its first sublayer
        row_ops.append(("copy", t) if t == start else ("acc", t - 1, t))
        # blocks before k end at ends[:k]; row t is block k's sum up to t
        sites.append([0] + ends[:k] + [t])
    return {"ends": ends, "row_ops": row_ops, "sites": sites}

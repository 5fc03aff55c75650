"""Exchange plans for running the same collectives across R real GPUs (host logic only).

On one GPU the library reads every contributor's gradients in place, because all R ranks are
buffers in the same memory.  Across R GPUs the same results need one exchange step each
(TIDE: Fig. 2b, the reduce-scatter; Fig. 6a, its sums formed where the shard lives; Fig. 5b, the
all-gather landing in parameter storage):

* reduce-scatter: GPU d pulls, from every contributor r, the slice of each parameter it will own,
  elements [d*s_p, d*s_p + v(d,p)*L_p) of g_r,p, into staging slot r at the slice's shard offset
  o_p; it then sums its R staging slots in ascending rank order into its fp32 shard
  (``tide_reduce_scatter_slots``), so the result is the single-GPU result bit for bit;
* all-gather: GPU d pulls, from every source rank r, the valid rows of each parameter piece,
  elements [o_p, o_p + v(r,p)*L_p) of shard_r, straight to element r*s_p of its parameter p.

Each plan entry is one contiguous copy (a peer cudaMemcpyAsync, or a range of plain peer loads
inside the summing kernel).  Contributors are visited in the order d+1, d+2, ..., d-1 (then d
itself, a local read), so that at any step the R destinations pull from R different sources.
The layout numbers come from the library's own planner (``tide_plan_layout``), the same ones the
kernels use.
"""
from __future__ import annotations

from typing import List, NamedTuple, Sequence


class Copy(NamedTuple):
    src_rank: int  # rank whose buffer is read
    param: int  # parameter p
    src_off: int  # element offset in the source buffer (gradient g_r,p, or shard_r)
    dst_off: int  # element offset in the destination buffer (staging slot, or parameter p)
    elems: int  # elements copied (bf16)


def source_order(R: int, d: int) -> List[int]:
    """Contributors in the order destination d visits them: d+1, ..., R-1, 0, ..., d."""
    return [(d + k) % R for k in range(1, R + 1)]


def _layout(R: int, rows: Sequence[int], row_len: Sequence[int]):
    from . import tide_plan_layout

    m, s, o, S, U = tide_plan_layout(R, list(rows), list(row_len))
    v = [[min(m[p], max(0, rows[p] - d * m[p])) for p in range(len(rows))] for d in range(R)]
    return m, s, o, S, v


def reduce_scatter_pulls(R: int, rows: Sequence[int], row_len: Sequence[int], d: int) -> List[Copy]:
    """Copies destination rank d makes for the reduce-scatter: from every contributor r, slice d
    of every parameter into staging slot r (a packed bf16 shard of S elements) at o_p.  Padding
    rows are not copied; the summing step writes +0.0f there."""
    m, s, o, S, v = _layout(R, rows, row_len)
    out = []
    for r in source_order(R, d):
        for p in range(len(rows)):
            n = v[d][p] * row_len[p]
            if n:
                out.append(Copy(r, p, d * s[p], o[p], n))
    return out


def all_gather_pulls(R: int, rows: Sequence[int], row_len: Sequence[int], d: int) -> List[Copy]:
    """Copies destination rank d makes for the all-gather: the valid rows of every source rank's
    piece of every parameter, from shard_r at o_p to parameter p at r*s_p."""
    m, s, o, S, v = _layout(R, rows, row_len)
    out = []
    for r in source_order(R, d):
        for p in range(len(rows)):
            n = v[r][p] * row_len[p]
            if n:
                out.append(Copy(r, p, o[p], r * s[p], n))
    return out

"""The layout-converting ("stock") path that the layout-aware collectives replace, on one GPU.

This is the comparison arm, not part of the TIDE path: plain PyTorch ops that emulate what FSDP2
does around its collectives (TIDE: Table 1, the full-group pack row; Table 7, the copy-out
columns; Table 8, whose stock numbers include the pack).  With R ranks emulated as R buffers on one
GPU:

* reduce-scatter: every contributor packs its per-parameter bf16 gradients into a full-group fp32
  buffer of R padded dim-0 chunks (``torch._chunk_cat``, as FSDP2 does; zero padding), and the R
  packed buffers are summed element-wise (``torch.sum`` over the contributor axis), which gives
  every destination rank's fp32 shard at once;
* all-gather copy-out: the gathered output, R packed bf16 shards back to back, is copied into
  padded per-parameter storage (``torch.split_with_sizes_copy``), whose first rows_p*L_p elements
  are the parameter.

``torch.sum`` fixes no summation order, so its shards agree with an ascending-rank fp32 sum only to
within rounding (|err| <= 2^-20 * sum_r |g_r| per element for the rank counts used here); the
copy-out is a bit copy.
"""
from __future__ import annotations

from typing import List, Sequence

import torch


class StockPath:
    """Buffers and ops of the stock path for one group: ``R`` ranks, parameters of shapes
    ``(rows_p, row_len_p)`` on ``device``.  The full-group buffer it needs is ``R*R*S*4`` bytes."""

    def __init__(self, R: int, rows: Sequence[int], row_len: Sequence[int], device):
        self.R = R
        self.rows = list(rows)
        self.row_len = list(row_len)
        self.P = len(self.rows)
        # padded rows per rank (torch.chunk / FSDP2 dim-0 split) and per-rank piece sizes
        self.m = [(r + R - 1) // R for r in self.rows]
        self.sizes = [self.m[p] * self.row_len[p] for p in range(self.P)]
        self.S = sum(self.sizes)
        self.device = torch.device(device)
        self.packed = torch.empty(R, R, self.S, dtype=torch.float32, device=self.device)
        self.padded = [torch.empty(R, n, dtype=torch.bfloat16, device=self.device) for n in self.sizes]
        self.have_chunk_cat = hasattr(torch, "_chunk_cat")

    @property
    def extra_buffer_bytes(self) -> int:
        """Bytes of the full-group pack buffers (the layout-aware path needs none)."""
        return self.packed.numel() * self.packed.element_size()

    def _pack(self, r: int, grads_r: Sequence[torch.Tensor]) -> None:
        views = [grads_r[p].view(torch.bfloat16).view(self.rows[p], self.row_len[p]) for p in range(self.P)]
        if self.have_chunk_cat:
            torch._chunk_cat(views, 0, self.R, out=self.packed[r])
            return
        # the same layout by hand: chunk d of every parameter, zero-padded, concatenated
        self.packed[r].zero_()
        o = 0
        for p in range(self.P):
            for d, piece in enumerate(torch.chunk(views[p], self.R, dim=0)):
                self.packed[r, d, o:o + piece.numel()].copy_(piece.reshape(-1))
            o += self.sizes[p]

    def reduce_scatter(self, grads: Sequence[Sequence[torch.Tensor]], out: torch.Tensor) -> torch.Tensor:
        """``grads[r][p]``: rank r's bf16 gradient of parameter p (any 16-bit dtype view);
        ``out``: [R, S] fp32, row d = destination rank d's shard.  Returns ``out``."""
        for r in range(self.R):
            self._pack(r, grads[r])
        torch.sum(self.packed, dim=0, out=out)
        return out

    def copy_out(self, gathered: torch.Tensor) -> List[torch.Tensor]:
        """``gathered``: [R, S] bf16, the all-gather output.  Returns the padded per-parameter
        tensors ([R, m_p*L_p] each); parameter p is the first rows_p*L_p elements of entry p."""
        torch.split_with_sizes_copy(gathered.view(torch.bfloat16).view(self.R, self.S), self.sizes, dim=1,
                                    out=self.padded)
        return self.padded

    def param_view(self, p: int) -> torch.Tensor:
        """Parameter p inside its padded copy-out storage (the valid rows only)."""
        return self.padded[p].view(-1)[: self.rows[p] * self.row_len[p]]

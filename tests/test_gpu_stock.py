"""GPU parity of the one-GPU stock comparator (the layout-converting path) against the CPU oracle.

The comparator packs every contributor's gradients into a full-group fp32 buffer and sums the
packed buffers with ``torch.sum``, whose summation order is not fixed: its shards are compared with
the oracle's exact (fp64) sum element by element within 2^-20 * sum_r |g_r| (the bound for any
order at these rank counts), padding exactly +0.  Its copy-out is a bit copy: every parameter inside
the padded copy-out storage must equal the oracle's all-gather bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import group, rng

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def stock():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from all_gather_tide_gb300 import stock as s

    return s


def groups():
    return [group("llama8b").scaled(16), group("qwen3moe").scaled(16), group("llama70b").scaled(32),
            group("wan_r8").scaled(8), group("wan_r16").scaled(8), group("wan_r32").scaled(16),
            group("wan_r64").scaled(16)]


@pytest.mark.parametrize("g", groups(), ids=[g.name for g in groups()])
def test_stock_reduce_scatter_within_bound_of_exact_sum(stock, g):
    lay = oracle.plan(g.R, g.rows, g.row_len)
    host = rng.group_grads(g)
    bits = [[t.numpy().view(np.uint16) for t in row] for row in host]
    exact = np.stack(oracle.exact_sum(lay, bits))
    # sum_r |g_r| per output element: the exact sum of the inputs with their sign bits cleared
    absum = np.stack(oracle.exact_sum(lay, [[b & np.uint16(0x7FFF) for b in row] for row in bits]))
    sp = stock.StockPath(g.R, g.rows, g.row_len, "cuda")
    assert sp.S == lay.S
    out = torch.full((g.R, lay.S), float("nan"), device="cuda")
    sp.reduce_scatter([[t.cuda() for t in row] for row in host], out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    err = np.abs(got - exact)
    bound = 2.0 ** -20 * absum
    bad = np.nonzero(~(err <= bound))
    assert bad[0].size == 0, f"{g.name}: {bad[0].size} elements outside the bound, e.g. {list(zip(*bad))[:4]}"
    pad = absum == 0
    assert np.all(out.view(torch.int32).cpu().numpy()[pad] == 0), "padding must be +0.0"


@pytest.mark.parametrize("g", groups(), ids=[g.name for g in groups()])
def test_stock_copy_out_matches_oracle_all_gather(stock, g):
    lay = oracle.plan(g.R, g.rows, g.row_len)
    shards = np.stack([rng.shard_bits(g, r, lay.S).numpy().view(np.uint16) for r in range(g.R)])
    want = oracle.all_gather(lay, list(shards), [np.zeros(g.numel(p), np.uint16) for p in range(g.P)])
    sp = stock.StockPath(g.R, g.rows, g.row_len, "cuda")
    sp.copy_out(torch.from_numpy(shards.view(np.int16)).cuda())
    torch.cuda.synchronize()
    for p in range(g.P):
        got = sp.param_view(p).view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, want[p]), f"{g.name}: parameter {p} differs"

"""tide_reduce_scatter_noalloc, the reduce-scatter for callers that cannot allocate memory.

Some callers cannot call cudaMalloc: a framework whose caching allocator already holds nearly all
device memory, or a communication path running beside compute that cannot afford the device-wide
synchronisation cudaMalloc/cudaFree may cause.  For them the library offers one entry point that
keeps its work tables in a fixed device array it carries instead of allocating.  This file checks,
through the C ABI, that its output equals the CPU oracle's and the group entry point's bit for bit
(the tolerance every reduce-scatter parity test here uses: the kernels keep the oracle's
ascending-rank fp32 order), on two calls in a row with different groups, with canary bands around
every buffer and sentinel-filled outputs; and that a group too large for the array is rejected
before anything runs.  It sits last in collection order so a run that stops at the first failure
has already run everything else; it also passes alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from workloads import Group, group, rng

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of canary before and after every buffer
CANARY = 0x5A
F32_SENTINEL = -1  # 0xFFFFFFFF: a NaN pattern no sum of these inputs produces


@pytest.fixture(scope="module")
def tide():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import all_gather_tide_gb300 as t

    t.lib()
    return t


class Banded:
    """A device buffer with canary bytes around the payload; `shift` elements of extra offset
    make the payload start off a 16-byte boundary."""

    def __init__(self, numel, dtype, shift=0):
        es = torch.tensor([], dtype=dtype).element_size()
        g = GUARD // es
        self.buf = torch.empty(2 * g + numel + shift, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(CANARY)
        self.lo, self.hi = g + shift, g + shift + numel
        self.view = self.buf[self.lo:self.hi]

    def intact(self) -> bool:
        b = self.buf.view(torch.uint8)
        es = self.buf.element_size()
        return bool((b[: self.lo * es] == CANARY).all()) and bool((b[self.hi * es:] == CANARY).all())


def _noalloc(tide, g, grads, shards, stream):
    """Direct C-ABI call of tide_reduce_scatter_noalloc; returns its status."""
    L = tide.lib()
    i64 = lambda xs: (ctypes.c_int64 * len(xs))(*xs)
    gp = (ctypes.c_void_p * (g.R * g.P))(*[t.data_ptr() for row in grads for t in row])
    sp = (ctypes.c_void_p * g.R)(*[s.data_ptr() for s in shards])
    return L.tide_reduce_scatter_noalloc(g.R, g.P, i64(g.rows), i64(g.row_len), gp, sp, stream.cuda_stream)


def test_noalloc_matches_oracle_and_group_entry_point_twice(tide):
    stream = torch.cuda.Stream()
    cases = [
        (group("qwen3moe").scaled(16), 0),
        (group("wan_r64").scaled(16), 0),
        # odd prefix offsets and gradients off a 16-byte boundary: the element-wise path
        (Group("odd-offsets", 3, (("a", 7, 5), ("b", 1, 1), ("c", 11, 3), ("d", 300, 17))), 1),
    ]
    runs = []
    for g, shift in cases:
        lay = oracle.plan(g.R, g.rows, g.row_len)
        host = rng.group_grads(g)
        want = oracle.reduce_scatter(lay, [[t.numpy().view(np.uint16) for t in row] for row in host])
        grads = [[Banded(t.numel(), torch.int16, shift) for t in row] for row in host]
        for row, hrow in zip(grads, host):
            for x, t in zip(row, hrow):
                x.view.copy_(t)
        shards = [Banded(lay.S, torch.float32) for _ in range(g.R)]
        for s in shards:
            s.view.view(torch.int32).fill_(F32_SENTINEL)
        runs.append((g, lay, want, grads, shards))
    torch.cuda.synchronize()
    # the calls follow one another on one stream with no synchronisation between them: each
    # call's tables replace the previous call's in the shared array only after the previous
    # kernel has read them
    for g, lay, want, grads, shards in runs:
        st = _noalloc(tide, g, [[x.view for x in row] for row in grads], [s.view for s in shards], stream)
        assert st == tide.TIDE_OK, tide.tide_strerror(st)
    stream.synchronize()
    for g, lay, want, grads, shards in runs:
        for d in range(g.R):
            got = shards[d].view.view(torch.int32).cpu().numpy().view(np.uint32)
            bad = np.nonzero(got != want[d].view(np.uint32))[0]
            assert bad.size == 0, f"{g.name}: shard {d} differs from the oracle at {bad[:8]} (of {bad.size})"
            assert shards[d].intact(), f"{g.name}: shard {d} guard band overwritten"
        assert all(x.intact() for row in grads for x in row), f"{g.name}: a gradient guard band changed"
        # and the group entry point gives the same bits
        ref = torch.full((g.R, lay.S), float("nan"), device="cuda")
        G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
        G.reduce_scatter([[x.view for x in row] for row in grads], list(ref))
        torch.cuda.synchronize()
        G.close()
        for d in range(g.R):
            assert torch.equal(shards[d].view.view(torch.int32), ref[d].view(torch.int32)), (g.name, d)


def test_noalloc_rejects_tables_beyond_scratch(tide):
    # 64 ranks x 400 parameters: 64*400*56 B of pieces + 8*(64*400 + 64) B of pointers > 1 MiB
    R, P = 64, 400
    rows = [64] * P
    row_len = [8] * P
    L = tide.lib()
    i64 = lambda xs: (ctypes.c_int64 * len(xs))(*xs)
    # real buffers of the right sizes (one shared by all entries): nothing may run, but if it did,
    # it would stay inside them
    grad = torch.zeros(64 * 8, dtype=torch.bfloat16, device="cuda")
    shard = torch.full((P * 8,), 7.0, dtype=torch.float32, device="cuda")
    gp = (ctypes.c_void_p * (R * P))(*([grad.data_ptr()] * (R * P)))
    sp = (ctypes.c_void_p * R)(*([shard.data_ptr()] * R))
    st = L.tide_reduce_scatter_noalloc(R, P, i64(rows), i64(row_len), gp, sp, None)
    assert st == tide.TIDE_ERANGE
    assert "range" in tide.tide_strerror(st)
    torch.cuda.synchronize()
    assert bool((shard == 7.0).all()), "a rejected call must not touch its outputs"

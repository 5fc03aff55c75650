"""tide_reduce_scatter_noalloc, the reduce-scatter for callers that cannot allocate memory.

Some callers cannot call cudaMalloc: a framework whose caching allocator already holds nearly all
device memory, or a communication path running beside compute that cannot afford the device-wide
synchronisation cudaMalloc/cudaFree may cause.  For them the library offers one entry point that
keeps its work tables in a fixed device array it carries instead of allocating.  This file checks,
through the C ABI, that its output equals the group entry point's (bit for bit, the tolerance all
reduce-scatter parity tests here use) on two calls in a row with different groups, and that a group
too large for the array is rejected before anything runs.  It sits last in collection order so a
run that stops at the first failure has already run everything else; it also passes alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import group, rng

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tide():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import all_gather_tide_gb300 as t

    t.lib()
    return t


def _noalloc(tide, g, grads, shards, stream):
    """Direct C-ABI call of tide_reduce_scatter_noalloc; returns its status."""
    L = tide.lib()
    i64 = lambda xs: (ctypes.c_int64 * len(xs))(*xs)
    gp = (ctypes.c_void_p * (g.R * g.P))(*[t.data_ptr() for row in grads for t in row])
    sp = (ctypes.c_void_p * g.R)(*[s.data_ptr() for s in shards])
    return L.tide_reduce_scatter_noalloc(g.R, g.P, i64(g.rows), i64(g.row_len), gp, sp, stream.cuda_stream)


def test_noalloc_matches_group_entry_point_twice(tide):
    stream = torch.cuda.Stream()
    cases = [group("qwen3moe").scaled(16), group("wan_r64").scaled(16)]
    inputs, outs = [], []
    for g in cases:
        grads = [[rng.grad_bits(g, r, p, device="cuda").view(torch.bfloat16) for p in range(g.P)]
                 for r in range(g.R)]
        S = tide.tide_plan_layout(g.R, g.rows, g.row_len)[3]
        out = torch.full((g.R, S), float("nan"), device="cuda")
        inputs.append(grads)
        outs.append(out)
    torch.cuda.synchronize()
    # two calls in a row on one stream, no synchronisation between them: the second call's tables
    # replace the first call's in the shared array only after the first kernel has read them
    for g, grads, out in zip(cases, inputs, outs):
        assert _noalloc(tide, g, grads, list(out), stream) == tide.TIDE_OK
    stream.synchronize()
    for g, grads, out in zip(cases, inputs, outs):
        ref = torch.full_like(out, float("nan"))
        G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
        G.reduce_scatter(grads, list(ref))
        torch.cuda.synchronize()
        G.close()
        a = out.view(torch.int32).cpu().numpy()
        b = ref.view(torch.int32).cpu().numpy()
        assert np.array_equal(a, b), f"{g.name}: no-alloc output differs from tide_reduce_scatter"


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
    shard = torch.zeros(P * 8, dtype=torch.float32, device="cuda")
    gp = (ctypes.c_void_p * (R * P))(*([grad.data_ptr()] * (R * P)))
    sp = (ctypes.c_void_p * R)(*([shard.data_ptr()] * R))
    st = L.tide_reduce_scatter_noalloc(R, P, i64(rows), i64(row_len), gp, sp, None)
    assert st == tide.TIDE_ERANGE
    assert "range" in tide.tide_strerror(st)

"""The multi-GPU exchange plans executed between real processes (gloo on the CPU, world size 2
and 3): every rank pulls exactly its slices, in the planned order, and the results match the
oracle's single-process reduce-scatter and all-gather bit for bit.

The local summing step, which on GPUs is the library's kernel over the staging slots
(tide_reduce_scatter_slots, checked against the oracle on a GPU in test_gpu_parity.py), is stood in
for here by torch fp32 adds in ascending rank order; what is tested here is the plan: which rank
sends which elements to whom, the offsets on both sides and the order of the exchange.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _group(R):
    from workloads import Group

    return Group("exchange", R, (("a", 5, 3), ("b", 7, 4), ("c", 2, 6), ("d", 33, 8), ("e", 1, 1)))


def _worker(rank, world, port, failures):
    try:
        import oracle
        from all_gather_tide_gb300 import exchange
        from workloads import rng

        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
        g = _group(world)
        lay = oracle.plan(g.R, g.rows, g.row_len)
        grads = [rng.grad_bits(g, rank, p).view(torch.int16).reshape(-1) for p in range(g.P)]

        # reduce-scatter: every destination's pull plan, run as sends from its sources
        staging = torch.zeros(world, lay.S, dtype=torch.int16)
        reqs, keep = [], []
        for d in range(world):
            for k, c in enumerate(exchange.reduce_scatter_pulls(g.R, g.rows, g.row_len, d)):
                if c.src_rank == rank and d != rank:
                    t = grads[c.param][c.src_off:c.src_off + c.elems].contiguous()
                    keep.append(t)
                    reqs.append(dist.isend(t, d, tag=k))
                elif d == rank and c.src_rank != rank:
                    buf = torch.empty(c.elems, dtype=torch.int16)
                    keep.append((buf, c))
                    reqs.append(dist.irecv(buf, c.src_rank, tag=k))
                elif d == rank:
                    staging[c.src_rank, c.dst_off:c.dst_off + c.elems] = grads[c.param][c.src_off:c.src_off + c.elems]
        for q in reqs:
            q.wait()
        for item in keep:
            if isinstance(item, tuple):
                buf, c = item
                staging[c.src_rank, c.dst_off:c.dst_off + c.elems] = buf
        # the local summing step: ascending rank, fp32
        wide = staging.view(torch.bfloat16).float()
        acc = wide[0].clone()
        for r in range(1, world):
            acc = acc + wide[r]
        all_grads = [[rng.grad_bits(g, r, p).numpy().view(np.uint16) for p in range(g.P)] for r in range(world)]
        want = oracle.reduce_scatter(lay, all_grads)[rank]
        if not np.array_equal(acc.numpy().view(np.uint32), want.view(np.uint32)):
            failures.append(f"rank {rank}: reduce-scatter shard differs")

        # all-gather: every destination pulls the valid rows of every source's shard
        shard = rng.shard_bits(g, rank, lay.S).view(torch.int16).reshape(-1)
        params = [torch.full((g.numel(p),), -1, dtype=torch.int16) for p in range(g.P)]
        reqs, keep = [], []
        for d in range(world):
            for k, c in enumerate(exchange.all_gather_pulls(g.R, g.rows, g.row_len, d)):
                if c.src_rank == rank and d != rank:
                    t = shard[c.src_off:c.src_off + c.elems].contiguous()
                    keep.append(t)
                    reqs.append(dist.isend(t, d, tag=10_000 + k))
                elif d == rank and c.src_rank != rank:
                    buf = torch.empty(c.elems, dtype=torch.int16)
                    keep.append((buf, c))
                    reqs.append(dist.irecv(buf, c.src_rank, tag=10_000 + k))
                elif d == rank:
                    params[c.param][c.dst_off:c.dst_off + c.elems] = shard[c.src_off:c.src_off + c.elems]
        for q in reqs:
            q.wait()
        for item in keep:
            if isinstance(item, tuple):
                buf, c = item
                params[c.param][c.dst_off:c.dst_off + c.elems] = buf
        shards = [rng.shard_bits(g, r, lay.S).numpy().view(np.uint16) for r in range(world)]
        ref = oracle.all_gather(lay, shards, [np.zeros(g.numel(p), np.uint16) for p in range(g.P)])
        for p in range(g.P):
            if not np.array_equal(params[p].numpy().view(np.uint16), ref[p]):
                failures.append(f"rank {rank}: parameter {p} differs after the all-gather")
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent, which fails the test
        failures.append(f"rank {rank}: {type(e).__name__}: {e}")


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_plans_between_processes(oracle_lib, world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    failures = mgr.list()
    mp.start_processes(_worker, args=(world, port, failures), nprocs=world, start_method="spawn", join=True)
    assert not list(failures), list(failures)


def test_exchange_plans_cover_every_element_once(oracle_lib):
    """Each destination's reduce-scatter pulls fill every valid element of its R staging slots
    exactly once, from the contributor that owns the slot, in the rotated source order; the
    all-gather pulls write every element of every parameter exactly once."""
    import oracle
    from all_gather_tide_gb300 import exchange

    for R in (1, 2, 3, 8):
        g = _group(R)
        lay = oracle.plan(g.R, g.rows, g.row_len)
        for d in range(R):
            cover = np.zeros((R, lay.S), np.int64)
            order = []
            for c in exchange.reduce_scatter_pulls(g.R, g.rows, g.row_len, d):
                cover[c.src_rank, c.dst_off:c.dst_off + c.elems] += 1
                assert c.src_off == d * int(lay.s[c.param]) and c.dst_off == int(lay.o[c.param])
                if not order or order[-1] != c.src_rank:
                    order.append(c.src_rank)
            assert order == [r for r in exchange.source_order(R, d) if r in order]
            for p in range(g.P):
                v = lay.valid_rows(d, p) * g.row_len[p]
                lo = int(lay.o[p])
                assert np.all(cover[:, lo:lo + v] == 1) and np.all(cover[:, lo + v:lo + int(lay.s[p])] == 0)
            seen = [np.zeros(g.numel(p), np.int64) for p in range(g.P)]
            for c in exchange.all_gather_pulls(g.R, g.rows, g.row_len, d):
                seen[c.param][c.dst_off:c.dst_off + c.elems] += 1
            assert all(np.all(s == 1) for s in seen)

"""Host-side logic of the benchmark: whole-job aggregation over replicas (world size 2, gloo on
the CPU), byte formulas, and the reference arm's JSON contract."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from workloads import group  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    ms = [40.0, 55.5][rank]
    m = bench.max_over_ranks(ms, world, "cpu")
    dist.barrier()
    out[rank] = m
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == out[1] == 55.5


def test_whole_job_value():
    # 2 replicas, 10 steps of 1 GB each, slowest rank 20 ms -> 1000 GB/s
    assert bench.whole_job_gbs(10**9, 10, 2, 20.0) == pytest.approx(1000.0)
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0


def test_byte_formulas_match_stated_sizes():
    import oracle

    g = group("llama70b")
    lay = oracle.plan(g.R, g.rows, g.row_len)
    assert bench.rs_bytes(g, lay.S, lay.U) == 8 * 855_654_400 * 2 + 8 * lay.S * 4
    assert abs(bench.rs_bytes(g, lay.S, lay.U) / 1e9 - 17.113) < 0.001
    assert bench.ag_bytes(lay.U) == 4 * 855_654_400


def test_reference_arm_json_contract():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--workload", "llama8b", "--scale", "8"], capture_output=True, text=True,
                         env=env, timeout=900)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the reference arm processes exactly the GPU arm's workload: same config dict
    g = group("llama8b").scaled(8)
    S, U = bench.layout(g)
    assert line["config"] == json.loads(json.dumps(bench.workload_config(g, S, U, 1)))


def test_host_oracle_baseline_covers_the_whole_group():
    g = group("llama8b").scaled(8)
    res = bench.cpu_baseline(g, None, passes=1)
    assert res["kind"] == "oracle" and res["unit"] == "GB/s" and res["value"] > 0 and res["one_thread_gbs"] > 0
    assert res["cores"] == len(os.sched_getaffinity(0))
    assert "whole" in res["sample"] and res["cpu_model"]


def test_host_oracle_parts_give_the_whole_group_result():
    """The threaded host baseline computes exactly the oracle's whole-group outputs."""
    import numpy as np

    import oracle

    g = group("qwen3moe").scaled(16)
    ho = bench.HostOracle(g, None)
    ho.time_passes(1, 0, 4)
    want = oracle.reduce_scatter(ho.lay, ho.grads)
    for d in range(g.R):
        assert np.array_equal(ho.out[d].view(np.uint32), want[d].view(np.uint32))
    params = oracle.all_gather(ho.lay, ho.shards, [np.zeros(g.numel(p), np.uint16) for p in range(g.P)])
    for p in range(g.P):
        assert np.array_equal(ho.params[p], params[p])


def test_mixed_bound_interpolates_between_probe_points():
    import bench

    rows = [{"copy_bytes": 73728, "read_gbs_per_sm": r, "write_gbs_per_sm": w}
            for r, w in [(150.0, 0.0), (120.0, 24.0), (50.0, 50.0)]]
    rows.append({"copy_bytes": 46080, "read_gbs_per_sm": 300.0, "write_gbs_per_sm": 0.0})  # other geometry: ignored
    per_sm, rd = bench.mixed_bound(rows, 0.0)
    assert (per_sm, rd) == (150.0, 150.0)
    per_sm, rd = bench.mixed_bound(rows, 0.2)  # exactly the second point
    assert abs(rd - 120.0) < 1e-9 and abs(per_sm - 144.0) < 1e-9
    per_sm, rd = bench.mixed_bound(rows, 0.6)  # halfway from ratio 0.2 to 1.0: reads halfway from 120 to 50
    assert abs(rd - 85.0) < 1e-9 and abs(per_sm - 85.0 * 1.6) < 1e-9
    assert bench.mixed_bound(rows, 1.5) == (None, None)

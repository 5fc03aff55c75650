"""The seeded input generator and the workload shapes (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import group, groups, rng


def _py_normal_bits(seed, rank, stream, i, sigma):
    """One element of the N(0, sigma) stand-in recomputed with Python ints and numpy fp32."""
    key = rng.stream_key(seed, rank, stream)
    k = 0
    for j in range(3):
        h = rng.splitmix_int(key, 3 * i + j)
        k += sum((h >> s) & 0xFFFF for s in (0, 16, 32, 48))
    x = np.float32(k - 393210) * np.float32(sigma / 65536.0)
    return int(torch.tensor([float(x)], dtype=torch.float32).to(torch.bfloat16).view(torch.int16)[0]) & 0xFFFF


def test_splitmix_reference_vector():
    # first outputs of SplitMix64 seeded with 0 (state 0), as published with the algorithm
    assert rng.splitmix_int(0, 0) == 0xE220A8397B1DCDAF
    assert rng.splitmix_int(0, 1) == 0x6E789E6AA1B965F4
    assert rng.splitmix_int(0, 2) == 0x06C45D188009454F


def test_uniform_int_matches_python_ints():
    t = rng.uniform_int_bf16_bits(3, 2, 5, 1000, -8, 8)
    vals = t.view(torch.bfloat16).float().numpy()
    key = rng.stream_key(3, 2, 5)
    for i in (0, 1, 17, 999):
        assert vals[i] == ((rng.splitmix_int(key, i) >> 32) % 17) - 8
    assert set(np.unique(vals).tolist()) == set(range(-8, 9))


def test_normal_matches_python_ints():
    t = rng.normal_bf16_bits(7, 1, 4, 500, 1e-3).numpy().astype(np.int64) & 0xFFFF
    for i in (0, 3, 250, 499):
        assert t[i] == _py_normal_bits(7, 1, 4, i, 1e-3)


def test_start_offset_is_a_slice():
    full = rng.normal_bf16_bits(1, 0, 0, 3000, 0.02)
    part = rng.normal_bf16_bits(1, 0, 0, 1000, 0.02, start=1500)
    assert torch.equal(full[1500:2500], part)


def test_normal_moments():
    x = rng.normal_bf16_bits(0, 0, 0, 1 << 20, 1e-3).view(torch.bfloat16).double()
    assert abs(x.mean().item()) < 1e-5
    assert abs(x.std().item() / 1e-3 - 1) < 0.01


def test_group_sizes():
    expect = {"tiny": (4, 3, 55), "llama8b": (8, 9, 218_112_000), "qwen3moe": (8, 393, 623_120_640),
              "llama70b": (8, 9, 855_654_400)}
    for name, (R, P, U) in expect.items():
        g = group(name)
        lay = oracle.plan(g.R, g.rows, g.row_len)
        assert (g.R, g.P, lay.U) == (R, P, U), name


@pytest.mark.parametrize("R,P", [(8, 3), (16, 6), (32, 10), (64, 21)])
def test_wan_sweep_fill_rule(R, P):
    """The written-out sweep lists follow the fill rule: extra matrix, then the DiT block cycled
    while each whole parameter still fits in 8,388,608 fp32 elements per rank, then one 1-D
    filler of R x remainder elements; every R pads."""
    g = group(f"wan_r{R}")
    assert g.R == R and g.P == P
    lay = oracle.plan(R, g.rows, g.row_len)
    assert lay.S == groups.WAN_SHARD_ELEMS
    # recompute the list with the oracle planner
    ps = [groups._WAN_EXTRA]
    i = 0
    while True:
        cand = groups._WAN_CYCLE[i % len(groups._WAN_CYCLE)]
        trial = oracle.plan(R, [p[1] for p in ps + [cand]], [p[2] for p in ps + [cand]])
        if trial.S > groups.WAN_SHARD_ELEMS:
            break
        ps.append(cand)
        i += 1
    rem = groups.WAN_SHARD_ELEMS - oracle.plan(R, [p[1] for p in ps], [p[2] for p in ps]).S
    assert [(r, l) for _, r, l in g.params[:-1]] == [(r, l) for _, r, l in ps]
    assert g.params[-1][1:] == (R * rem, 1)
    assert any(r % R for r in g.rows)


def test_positions_match_ranges():
    idx = torch.tensor([0, 5, 1234, 77, 2999])
    full = rng.normal_bf16_bits(2, 3, 4, 3000, 1e-3)
    assert torch.equal(rng.normal_bf16_bits(2, 3, 4, 0, 1e-3, idx=idx), full[idx])
    fi = rng.uniform_int_bf16_bits(2, 3, 4, 3000)
    assert torch.equal(rng.uniform_int_bf16_bits(2, 3, 4, 0, idx=idx), fi[idx])

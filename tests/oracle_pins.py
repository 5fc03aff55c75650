"""Pins of the CPU oracle against facts fixed outside it.

Each pin checks the oracle against something other than itself: hand-worked values (golden
files), closed forms of the layout, the library routines the definition reduces to
(``torch.chunk`` dim-0 sharding as in FSDP2, torch's bf16 -> fp32 conversion, torch fp32 adds in
ascending rank order), exact integer arithmetic, and invariants (all-gather of shard(x) is x;
padding is +0; the total over all shards equals the total gradient).  The set is chosen so that
a plausible slip anywhere in the oracle (a dropped term, a wrong sign, a wrong index, a transposed
operand, a wrong rounding of the padded rows) fails at least one of them; ``test_oracle_mutants``
plants such slips in copies of the oracle and checks exactly that.

Every pin raises ``AssertionError`` on failure.  "TIDE" is "The Endgame of FSDP Communication"
(arXiv 2610.38228); citations name its abstract, figures and tables.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from workloads import rng

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

JUNK_BF16 = 0xDEAD
SENTINEL_BF16 = 0xBEEF


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits16(a) -> np.ndarray:
    return np.asarray(a).astype(np.int64).astype(np.uint16)


def _f32_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def random_groups(seed: int, n: int = 6):
    """Small random groups: ragged rows, 1-D and 2-D parameters, R from 1 to 9."""
    rs = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        R = int(rs.integers(1, 10))
        P = int(rs.integers(1, 6))
        rows = [int(rs.integers(1, 3 * R + 4)) for _ in range(P)]
        row_len = [int(rs.choice([1, 2, 3, 5, 8, 13])) for _ in range(P)]
        out.append((R, rows, row_len))
    return out


def wide_bf16(seed: int, n: int, spread: int = 18) -> np.ndarray:
    """Random finite bf16 patterns with exponents spread over 2^-spread .. 2^spread: sums of a few
    of them need far more than fp32's 24 significant bits, but fewer than fp64's 53."""
    rs = np.random.default_rng(seed)
    x = (rs.standard_normal(n) * np.exp2(rs.integers(-spread, spread + 1, n))).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def random_bf16(seed: int, n: int, scale: float = 1.0) -> np.ndarray:
    """Random finite bf16 bit patterns with varied exponents (fold order matters for them)."""
    rs = np.random.default_rng(seed)
    x = (rs.standard_normal(n) * scale * np.exp2(rs.integers(-6, 6, n))).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------------------------
# independent constructions (torch.chunk = FSDP2's dim-0 split)


def chunk_pieces(R: int, x: torch.Tensor):
    """Rank d's piece of a tensor and its padded row count, from ``torch.chunk`` alone."""
    ch = torch.chunk(x, R, dim=0)
    m = ch[0].shape[0]
    return [ch[d] if d < len(ch) else x[:0] for d in range(R)], m


def torch_reduce_scatter(R, rows, row_len, grads):
    """Reference reduce-scatter from torch.chunk pieces, fp32 adds in ascending rank order."""
    shards = []
    pad_masks = []
    for d in range(R):
        parts, masks = [], []
        for p in range(len(rows)):
            pieces = []
            m = None
            for r in range(R):
                t = torch.from_numpy(grads[r][p].view(np.int16).copy()).view(torch.bfloat16)
                ps, m = chunk_pieces(R, t.reshape(rows[p], row_len[p]))
                pieces.append(ps[d].float())
            acc = pieces[0].clone()
            for r in range(1, R):
                acc = acc + pieces[r]
            valid = acc.shape[0]
            full = torch.zeros(m, row_len[p], dtype=torch.float32)
            full[:valid] = acc
            mask = torch.zeros(m, row_len[p], dtype=torch.bool)
            mask[valid:] = True
            parts.append(full.reshape(-1))
            masks.append(mask.reshape(-1))
        shards.append(torch.cat(parts).numpy())
        pad_masks.append(torch.cat(masks).numpy())
    return shards, pad_masks


def torch_pack(R, rows, row_len, params, junk):
    """Reference packing of per-parameter tensors into R shards; padding filled with ``junk``."""
    shards = []
    for d in range(R):
        parts = []
        for p in range(len(rows)):
            t = torch.from_numpy(params[p].view(np.int16).copy()).reshape(rows[p], row_len[p])
            ps, m = chunk_pieces(R, t)
            full = torch.full((m, row_len[p]), junk - 65536 if junk >= 32768 else junk, dtype=torch.int16)
            full[: ps[d].shape[0]] = ps[d]
            parts.append(full.reshape(-1))
        shards.append(torch.cat(parts).numpy().view(np.uint16))
    return shards


# ---------------------------------------------------------------------------------------------
# pins


def pin_plan_golden():
    """Planner on the tiny group equals the hand-derived Table 2 quantities."""
    g = _golden("tiny_plan.json")
    lay = oracle.plan(g["R"], g["rows"], g["row_len"])
    assert lay.m.tolist() == g["m"], lay.m
    assert lay.s.tolist() == g["s"], lay.s
    assert lay.o.tolist() == g["o"], lay.o
    assert (lay.S, lay.U) == (g["S"], g["U"])
    for p, vs in enumerate(g["valid_rows_by_param"]):
        assert [lay.valid_rows(d, p) for d in range(g["R"])] == vs, (p, vs)
    assert lay.R * lay.S - lay.U == g["padding_elements_total"]


def pin_hand_worked():
    """Reduce-scatter and all-gather of the hand-worked R=2 example, bit for bit."""
    g = _golden("hand_worked.json")
    R, rows, row_len = g["R"], g["rows"], g["row_len"]
    lay = oracle.plan(R, rows, row_len)

    def bf(vals):
        return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    grads = [[bf(g["grads"][f"rank{r}"][n]) for n in ("A", "B")] for r in range(R)]
    shards = oracle.reduce_scatter(lay, grads)
    for d in range(R):
        want = np.asarray(g["rs_shards"][d], np.float32)
        assert np.array_equal(_f32_bits(shards[d]), _f32_bits(want)), (d, shards[d], want)
    ag_in = [bf(s) for s in g["ag_shards"]]
    params = [np.full(rows[p] * row_len[p], SENTINEL_BF16, np.uint16) for p in range(len(rows))]
    oracle.all_gather(lay, ag_in, params)
    for p, n in enumerate(("A", "B")):
        assert np.array_equal(params[p], bf(g["ag_params"][n])), (n, params[p])


def pin_plan_closed_forms(seed: int = 1):
    """sum_d v(d,p) = rows_p; R*S - U = sum_p (R*m_p - rows_p)*L_p; m_p is the least row count
    with R*m_p >= rows_p; offsets are the prefix sums of s_p."""
    for R, rows, row_len in random_groups(seed, 40):
        lay = oracle.plan(R, rows, row_len)
        for p in range(lay.P):
            assert sum(lay.valid_rows(d, p) for d in range(R)) == rows[p]
            assert R * lay.m[p] >= rows[p] > R * (lay.m[p] - 1)
            assert lay.s[p] == lay.m[p] * row_len[p]
            assert lay.o[p] == sum(int(lay.s[q]) for q in range(p))
        assert lay.S == int(lay.s.sum())
        assert lay.U == sum(r * l for r, l in zip(rows, row_len))
        assert R * lay.S - lay.U == sum((R * int(lay.m[p]) - rows[p]) * row_len[p] for p in range(lay.P))


def pin_pack_vs_torch_chunk(seed: int = 2):
    """The oracle's shard packing equals torch.chunk dim-0 pieces padded and concatenated."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed)):
        lay = oracle.plan(R, rows, row_len)
        params = [random_bf16(seed * 100 + gi * 10 + p, rows[p] * row_len[p]) for p in range(len(rows))]
        shards = [np.full(lay.S, JUNK_BF16, np.uint16) for _ in range(R)]
        oracle.shard_bf16(lay, params, shards)
        want = torch_pack(R, rows, row_len, params, JUNK_BF16)
        for d in range(R):
            assert np.array_equal(shards[d], want[d]), (R, rows, row_len, d)


def pin_rs_vs_torch_chunk(seed: int = 3):
    """Reduce-scatter equals torch.chunk pieces summed with torch fp32 adds in ascending rank
    order, padding zero-filled (random varied-exponent values, so the fold order shows)."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed)):
        lay = oracle.plan(R, rows, row_len)
        grads = [[random_bf16(seed * 1000 + gi * 100 + r * 10 + p, rows[p] * row_len[p])
                  for p in range(len(rows))] for r in range(R)]
        got = oracle.reduce_scatter(lay, grads)
        want, pad = torch_reduce_scatter(R, rows, row_len, grads)
        for d in range(R):
            assert np.array_equal(_f32_bits(got[d]), _f32_bits(want[d])), (R, rows, row_len, d)
            assert np.all(_f32_bits(got[d])[pad[d]] == 0), "padding must be +0.0"


def pin_rs_integer_exact(seed: int = 4):
    """Integer-valued bf16 inputs in [-8, 8]: every fp32 partial sum is an exact integer, so the
    result equals the exact integer sum (computed with Python ints) in any order."""
    for R, rows, row_len in random_groups(seed) + [(4, [5, 7, 2], [3, 4, 6])]:
        lay = oracle.plan(R, rows, row_len)
        grads = [[rng.uniform_int_bf16_bits(seed, r, p, rows[p] * row_len[p]).numpy().view(np.uint16)
                  for p in range(len(rows))] for r in range(R)]
        ints = [[torch.from_numpy(grads[r][p].view(np.int16).copy()).view(torch.bfloat16).float().numpy()
                 .astype(np.int64) for p in range(len(rows))] for r in range(R)]
        got = oracle.reduce_scatter(lay, grads)
        exact = oracle.exact_sum(lay, grads)
        for d in range(R):
            assert np.array_equal(got[d].astype(np.float64), exact[d])
            for p in range(len(rows)):
                m, L = int(lay.m[p]), row_len[p]
                for j in range(m):
                    row = d * m + j
                    for k in range(L):
                        want = sum(int(ints[r][p][row * L + k]) for r in range(R)) if row < rows[p] else 0
                        assert got[d][int(lay.o[p]) + j * L + k] == want


def pin_total_sum(seed: int = 5):
    """Sum over all destination shards = sum of all gradients: exact in fp64 for integer inputs,
    within (R-1) * 2^-24 * sum|g| for real-valued inputs (fp32 left-fold error bound)."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed)):
        lay = oracle.plan(R, rows, row_len)
        for kind in ("int", "real"):
            if kind == "int":
                grads = [[rng.uniform_int_bf16_bits(seed + gi, r, p, rows[p] * row_len[p]).numpy().view(np.uint16)
                          for p in range(len(rows))] for r in range(R)]
            else:
                grads = [[random_bf16(seed * 7 + gi * 100 + r * 10 + p, rows[p] * row_len[p])
                          for p in range(len(rows))] for r in range(R)]
            widened = [oracle.bf16_to_f32(grads[r][p]).astype(np.float64) for r in range(R) for p in range(len(rows))]
            total_in = math.fsum(float(v) for a in widened for v in a)
            abs_in = math.fsum(float(abs(v)) for a in widened for v in a)
            shards = oracle.reduce_scatter(lay, grads)
            total_out = math.fsum(float(v) for s in shards for v in s.astype(np.float64))
            if kind == "int":
                assert total_out == total_in
            else:
                assert abs(total_out - total_in) <= (R - 1) * 2.0 ** -24 * abs_in + 1e-300


def pin_single_rank_is_widening(seed: int = 6):
    """R = 1: the only shard is every parameter widened to fp32 (torch's bf16 -> fp32), concatenated."""
    for _, rows, row_len in random_groups(seed):
        lay = oracle.plan(1, rows, row_len)
        params = [random_bf16(seed + p, rows[p] * row_len[p]) for p in range(len(rows))]
        got = oracle.reduce_scatter(lay, [params])[0]
        want = torch.cat([torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).float() for a in params])
        assert np.array_equal(_f32_bits(got), _f32_bits(want.numpy()))


def pin_bf16_widening():
    """The oracle's bf16 -> fp32 widening equals torch's for all 65536 bit patterns."""
    L = oracle.lib()
    bits = np.arange(65536, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([L.oracle_bf16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(_f32_bits(got)[~nan], _f32_bits(want)[~nan])


def pin_negative_zero():
    """Reading: the fold starts from rank 0's value, so an all -0.0 sum stays -0.0 and a mixed
    -0.0 / +0.0 sum is +0.0 (IEEE round-to-nearest)."""
    lay = oracle.plan(3, [3], [1])
    nz, pz = 0x8000, 0x0000
    grads = [[np.array(v, np.uint16)] for v in ([nz, nz, pz], [nz, pz, nz], [nz, nz, nz])]
    out = oracle.reduce_scatter(lay, grads)
    assert _f32_bits(out[0])[0] == 0x80000000 and _f32_bits(out[1])[0] == 0 and _f32_bits(out[2])[0] == 0


def pin_ag_roundtrip(seed: int = 7):
    """all_gather(shard(x)) == x bit for bit, junk padding never reaches the output, and the
    all-gather equals the inverse of torch.chunk packing."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed)):
        lay = oracle.plan(R, rows, row_len)
        x = [random_bf16(seed * 31 + gi * 7 + p, rows[p] * row_len[p], 0.02) for p in range(len(rows))]
        shards = torch_pack(R, rows, row_len, x, JUNK_BF16)
        out = [np.full(rows[p] * row_len[p], SENTINEL_BF16, np.uint16) for p in range(len(rows))]
        oracle.all_gather(lay, shards, out)
        for p in range(len(rows)):
            assert np.array_equal(out[p], x[p]), (R, rows, row_len, p)
            assert not np.any(out[p] == JUNK_BF16)
        packed = [np.full(lay.S, JUNK_BF16, np.uint16) for _ in range(R)]
        oracle.shard_bf16(lay, x, packed)
        back = [np.full(rows[p] * row_len[p], SENTINEL_BF16, np.uint16) for p in range(len(rows))]
        oracle.all_gather(lay, packed, back)
        for p in range(len(rows)):
            assert np.array_equal(back[p], x[p])


def pin_rs_points(seed: int = 8):
    """Single-output evaluation equals the full reduce-scatter at every position."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed)):
        lay = oracle.plan(R, rows, row_len)
        grads = [[random_bf16(seed * 1000 + gi * 100 + r * 10 + p, rows[p] * row_len[p])
                  for p in range(len(rows))] for r in range(R)]
        full = oracle.reduce_scatter(lay, grads)
        d = np.repeat(np.arange(R), lay.S)
        j = np.tile(np.arange(lay.S), R)
        pts = oracle.rs_points(lay, d, j, lambda r, p, idx: grads[r][p][idx])
        assert np.array_equal(_f32_bits(pts), _f32_bits(np.concatenate(full)))


def pin_exact_sum_vs_fsum(seed: int = 10):
    """The fp64 reference sum equals math.fsum (Shewchuk's exactly rounded sum) of the widened
    inputs at every output position, with +0 in padding.  The inputs' exponents span 2^-18 .. 2^18,
    so an exact sum needs up to ~45 significant bits: fp64 keeps them all, an fp32 accumulator or a
    dropped term does not."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed) + [(9, [4, 11], [7, 3])]):
        lay = oracle.plan(R, rows, row_len)
        grads = [[wide_bf16(seed * 1000 + gi * 100 + r * 10 + p, rows[p] * row_len[p])
                  for p in range(len(rows))] for r in range(R)]
        widened = [[oracle.bf16_to_f32(grads[r][p]).astype(np.float64) for p in range(len(rows))] for r in range(R)]
        exact = oracle.exact_sum(lay, grads)
        for d in range(R):
            for p in range(len(rows)):
                m, L = int(lay.m[p]), row_len[p]
                for j in range(m):
                    row = d * m + j
                    for k in range(L):
                        got = exact[d][int(lay.o[p]) + j * L + k]
                        if row < rows[p]:
                            want = math.fsum(float(widened[r][p][row * L + k]) for r in range(R))
                            assert got == want, (R, rows, row_len, d, p, j, k, got, want)
                        else:
                            assert got == 0.0 and not math.copysign(1.0, got) < 0


def pin_parts_partition_the_group(seed: int = 11):
    """The per-(rank, parameter-range) parts write exactly their own elements (everything else keeps
    its sentinel), and all parts together give the whole-group result bit for bit, for the
    reduce-scatter and the all-gather alike."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed)):
        lay = oracle.plan(R, rows, row_len)
        P = len(rows)
        grads = [[random_bf16(seed * 1000 + gi * 100 + r * 10 + p, rows[p] * row_len[p])
                  for p in range(P)] for r in range(R)]
        full = oracle.reduce_scatter(lay, grads)
        out = [np.full(lay.S, np.nan, np.float32) for _ in range(R)]
        m = oracle.marshal_reduce_scatter(lay, grads, out)
        for d in range(R):
            for p in range(P):
                before = [o.copy() for o in out]
                oracle.reduce_scatter_part(m, d, p, p + 1)
                lo, hi = int(lay.o[p]), int(lay.o[p] + lay.s[p])
                for e in range(R):
                    changed = _f32_bits(out[e]) != _f32_bits(before[e])
                    if e != d:
                        assert not changed.any()
                    else:
                        assert not changed[:lo].any() and not changed[hi:].any()
                        assert np.array_equal(_f32_bits(out[e][lo:hi]), _f32_bits(full[e][lo:hi]))
        for d in range(R):
            assert np.array_equal(_f32_bits(out[d]), _f32_bits(full[d]))
        shards = [random_bf16(seed * 100 + gi * 10 + r, lay.S, 0.02) for r in range(R)]
        want = oracle.all_gather(lay, shards, [np.full(rows[p] * row_len[p], SENTINEL_BF16, np.uint16)
                                               for p in range(P)])
        got = [np.full(rows[p] * row_len[p], SENTINEL_BF16, np.uint16) for p in range(P)]
        ma = oracle.marshal_all_gather(lay, shards, got)
        for r in range(R):
            oracle.all_gather_part(ma, r, 0, P)
            for p in range(P):
                v = lay.valid_rows(r, p) * row_len[p]
                lo = r * int(lay.m[p]) * row_len[p]
                assert np.array_equal(got[p][lo:lo + v], want[p][lo:lo + v])
                assert np.all(got[p][lo + v:] == SENTINEL_BF16)  # later ranks' rows not yet written
        for p in range(P):
            assert np.array_equal(got[p], want[p])


ALL_PINS = [
    pin_plan_golden,
    pin_hand_worked,
    pin_plan_closed_forms,
    pin_pack_vs_torch_chunk,
    pin_rs_vs_torch_chunk,
    pin_rs_integer_exact,
    pin_total_sum,
    pin_single_rank_is_widening,
    pin_bf16_widening,
    pin_negative_zero,
    pin_ag_roundtrip,
    pin_rs_points,
    pin_exact_sum_vs_fsum,
    pin_parts_partition_the_group,
]


def pin_ag_points(seed: int = 9):
    """Single-output all-gather source positions reproduce the full all-gather."""
    for gi, (R, rows, row_len) in enumerate(random_groups(seed)):
        lay = oracle.plan(R, rows, row_len)
        shards = [random_bf16(seed * 100 + gi * 10 + r, lay.S, 0.02) for r in range(R)]
        out = [np.full(rows[p] * row_len[p], SENTINEL_BF16, np.uint16) for p in range(len(rows))]
        oracle.all_gather(lay, shards, out)
        for p in range(len(rows)):
            idx = np.arange(rows[p] * row_len[p])
            r, j = oracle.ag_points(lay, p, idx)
            got = np.array([shards[a][b] for a, b in zip(r, j)], np.uint16)
            assert np.array_equal(got, out[p])


ALL_PINS.append(pin_ag_points)

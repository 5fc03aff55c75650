"""GPU parity of the CUDA path (called through the C ABI) against the CPU oracle.

Reduced-size groups (the workload parameter lists with every dimension divided down, plus edge
groups) are compared element by element, bit for bit, with 4 KiB canary guard bands around every
device buffer and sentinel-prefilled outputs (so every output element must be written and every
padding element must come out +0.0).  Full-size groups run in the launch configuration the
benchmark times (default CTA counts) and are checked on sampled outputs that the oracle computes
one by one from regenerated inputs, plus properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
from workloads import Group, group, rng

pytestmark = pytest.mark.gpu

GUARD_BYTES = 4096
CANARY = 0x5A
F32_SENTINEL = -1  # 0xFFFFFFFF, a NaN pattern no sum produces here
BF16_SENTINEL = 0xBEEF - 65536
BF16_JUNK = 0xDEAD - 65536


@pytest.fixture(scope="module")
def tide():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import all_gather_tide_gb300 as t

    t.lib()
    return t


class Guarded:
    """A device buffer with canary bytes before and after the payload view."""

    def __init__(self, numel, dtype, fill=None, offset_elems=0, src=None):
        es = torch.tensor([], dtype=dtype).element_size()
        g = GUARD_BYTES // es
        self.buf = torch.empty(2 * g + numel + offset_elems, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(CANARY)
        self.lo, self.hi = g + offset_elems, g + offset_elems + numel
        self.view = self.buf[self.lo:self.hi]
        if src is not None:
            self.view.copy_(src)
        elif fill is not None:
            self.view.view(torch.int32 if es == 4 else torch.int16).fill_(fill)

    def guards_intact(self) -> bool:
        b = self.buf.view(torch.uint8)
        es = self.buf.element_size()
        head = b[: self.lo * es]
        tail = b[self.hi * es:]
        return bool((head == CANARY).all()) and bool((tail == CANARY).all())


def f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def edge_groups():
    return [
        Group("single-rank", 1, (("a", 37, 5), ("b", 1024, 8), ("c", 3, 1))),
        Group("one-row-64-ranks", 64, (("a", 1, 4096), ("b", 3, 8), ("c", 100, 1), ("d", 65, 3))),
        Group("odd-offsets", 3, (("a", 7, 5), ("b", 1, 1), ("c", 11, 3), ("d", 300, 17))),
        Group("ragged-tails", 8, (("a", 1001, 8), ("b", 13, 24), ("c", 40097, 1), ("d", 9, 4104))),
        Group("integer-r16", 16, (("a", 333, 64), ("b", 64, 512), ("c", 17, 1)), grad_kind="int"),
    ]


def reduced_groups():
    return [
        group("tiny"),
        group("llama8b").scaled(16),
        group("qwen3moe").scaled(16),
        group("llama70b").scaled(32),
        group("wan_r8").scaled(8),
        group("wan_r16").scaled(8),
        group("wan_r32").scaled(16),
        group("wan_r64").scaled(16),
    ] + edge_groups()


def _ids(gs):
    return [g.name for g in gs]


def run_rs(tide, g, ctas=0, misalign=False, flags=0, variant=0):
    lay = oracle.plan(g.R, g.rows, g.row_len)
    host = rng.group_grads(g)
    want = oracle.reduce_scatter(lay, [[t.numpy().view(np.uint16) for t in row] for row in host])
    off = 1 if misalign else 0
    grads = [[Guarded(t.numel(), torch.int16, src=t, offset_elems=off) for t in row] for row in host]
    shards = [Guarded(lay.S, torch.float32, fill=F32_SENTINEL) for _ in range(g.R)]
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), flags)
    G.set_ctas(ctas, 0)
    G.set_rs_variant(variant)
    G.reduce_scatter([[x.view for x in row] for row in grads], [s.view for s in shards])
    torch.cuda.synchronize()
    assert G.device_status() == 0
    for d in range(g.R):
        got = f32_bits(shards[d].view)
        bad = np.nonzero(got != want[d].view(np.uint32))[0]
        assert bad.size == 0, f"{g.name}: shard {d} differs at {bad[:8]} (of {bad.size})"
        assert shards[d].guards_intact(), f"{g.name}: shard {d} guard band overwritten"
    for row in grads:
        for x in row:
            assert x.guards_intact()
    G.close()


def run_ag(tide, g, ce=False, ctas=0, misalign=False, uniform=True, flags=0, variant=0, bands=1):
    lay = oracle.plan(g.R, g.rows, g.row_len)
    host = []
    for r in range(g.R):
        s = rng.shard_bits(g, r, lay.S).numpy().copy()
        for p in range(g.P):  # junk in every padding position
            v = lay.valid_rows(r, p) * int(lay.row_len[p])
            s[int(lay.o[p]) + v: int(lay.o[p] + lay.s[p])] = BF16_JUNK
        host.append(s)
    want = oracle.all_gather(lay, [h.view(np.uint16) for h in host],
                             [np.full(g.numel(p), BF16_SENTINEL & 0xFFFF, np.uint16) for p in range(g.P)])
    off = 1 if misalign else 0
    if uniform:
        packed = Guarded(g.R * lay.S, torch.int16, src=torch.from_numpy(np.concatenate(host)), offset_elems=off)
        shard_views = [packed.view[r * lay.S:(r + 1) * lay.S] for r in range(g.R)]
        guards = [packed]
    else:
        # one buffer, shards separated by growing gaps: no single pitch fits
        starts = [r * lay.S + 8 * r * (r + 1) // 2 for r in range(g.R)]
        packed = Guarded(starts[-1] + lay.S, torch.int16, fill=0, offset_elems=off)
        shard_views = [packed.view[a:a + lay.S] for a in starts]
        for v, h in zip(shard_views, host):
            v.copy_(torch.from_numpy(h))
        guards = [packed]
    params = [Guarded(g.numel(p), torch.int16, fill=BF16_SENTINEL, offset_elems=off) for p in range(g.P)]
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), flags)
    G.set_ctas(0, ctas)
    G.set_ag_variant(variant)
    G.set_ce_bands(bands)
    if ce:
        G.all_gather_ce(shard_views, [x.view for x in params])
    else:
        G.all_gather(shard_views, [x.view for x in params])
    torch.cuda.synchronize()
    assert G.device_status() == 0
    for p in range(g.P):
        got = params[p].view.cpu().numpy().view(np.uint16)
        bad = np.nonzero(got != want[p])[0]
        assert bad.size == 0, f"{g.name}: param {p} differs at {bad[:8]} (of {bad.size})"
        assert not np.any(got == (BF16_JUNK & 0xFFFF))
        assert params[p].guards_intact()
    for x in guards:
        assert x.guards_intact()
    copies = G.last_ce_copies() if ce else None
    G.close()
    return copies


# ---- reduced sizes, element by element -------------------------------------------------------


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_reduce_scatter_matches_oracle(tide, g):
    run_rs(tide, g)


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_reduce_scatter_bulk_matches_oracle(tide, g):
    run_rs(tide, g, variant=tide.TIDE_RS_BULK)


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_reduce_scatter_tmem_matches_oracle(tide, g):
    run_rs(tide, g, variant=tide.TIDE_RS_TMEM)


@pytest.mark.parametrize("ctas", [1, 3, 16, 152, 1000])
def test_reduce_scatter_tmem_cta_counts(tide, ctas):
    run_rs(tide, group("qwen3moe").scaled(16), ctas=ctas, variant=tide.TIDE_RS_TMEM)
    run_rs(tide, group("wan_r64").scaled(16), ctas=ctas, variant=tide.TIDE_RS_TMEM)
    run_rs(tide, edge_groups()[3], ctas=ctas, variant=tide.TIDE_RS_TMEM)


@pytest.mark.parametrize("ctas", [1, 3, 16, 24, 152])
def test_reduce_scatter_bulk_cta_counts(tide, ctas):
    run_rs(tide, group("qwen3moe").scaled(16), ctas=ctas, variant=tide.TIDE_RS_BULK)
    run_rs(tide, group("wan_r64").scaled(16), ctas=ctas, variant=tide.TIDE_RS_BULK)


SPECIAL_FINITE = [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080, 0x7F7F, 0xFF7F, 0x3F80, 0xBF80,
                  0x0100, 0x00FF]
SPECIAL_NONFINITE = [0x7F80, 0xFF80, 0x7FC0]


def _special_grads(g, seed, pool):
    rs = np.random.default_rng(seed)
    out = []
    for r in range(g.R):
        row = []
        for p in range(g.P):
            n = g.numel(p)
            base = rng.grad_bits(g, r, p).numpy().view(np.uint16).copy()
            pick = rs.random(n) < 0.5
            base[pick] = np.asarray(pool, np.uint16)[rs.integers(0, len(pool), int(pick.sum()))]
            row.append(base)
        out.append(row)
    for r in range(g.R):  # one element that is -0.0 on every rank: its sum must stay -0.0
        out[r][-1][0] = 0x8000
    return out


@pytest.mark.parametrize("variant", [1, 2, 3], ids=["register", "bulk", "tmem"])
def test_special_values(tide, variant):
    """Signed zeros, bf16 subnormals (fp32 subnormals after widening), the largest finite values
    (whose sums overflow to infinity under round-to-nearest), infinities and NaN: finite results
    bit for bit, NaN where the oracle has NaN."""
    g = Group("specials", 8, (("a", 640, 64), ("b", 37, 24), ("c", 4099, 1)))
    lay = oracle.plan(g.R, g.rows, g.row_len)
    for seed, pool in ((1, SPECIAL_FINITE), (2, SPECIAL_FINITE + SPECIAL_NONFINITE)):
        host = _special_grads(g, seed, pool)
        want = np.stack(oracle.reduce_scatter(lay, host))
        dev = [[torch.from_numpy(a.view(np.int16)).cuda() for a in row] for row in host]
        out = torch.empty(g.R, lay.S, dtype=torch.float32, device="cuda")
        G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
        G.set_rs_variant(variant)
        G.reduce_scatter(dev, list(out))
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
        if seed == 1:
            assert np.isinf(want).any() and (want.view(np.uint32) == 0x80000000).any()
            assert ((np.abs(want) < 1.1754944e-38) & (want != 0)).any()  # fp32 subnormal results
        G.close()


@pytest.mark.parametrize("variant", [2, 3], ids=["bulk", "tmem"])
def test_bulk_wait_timeout_reports_status_and_context_survives(tide, variant):
    """A producer that never signals (test hook) makes the bounded waits expire (the consumers'
    on data that never arrives, the producer's on stages never freed, the writers' on sums never
    handed over): the kernel returns, the status word records the first wait that gave up, and the
    next call runs normally."""
    g = group("llama70b").scaled(64)
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    G.set_rs_variant(variant)
    G.set_ctas(8, 0)
    G.set_wait_timeout(50_000_000)  # 50 ms
    grads = [[rng.grad_bits(g, r, p, device="cuda").view(torch.bfloat16) for p in range(g.P)] for r in range(g.R)]
    shards = torch.zeros(g.R, G.S, dtype=torch.float32, device="cuda")
    G.set_debug(tide.TIDE_DEBUG_STALL_PRODUCER)
    G.reduce_scatter(grads, list(shards))
    torch.cuda.synchronize()
    # every side waits on something nobody provides; whichever bound expires first is recorded
    assert G.device_status() in ((1, 2) if variant == 2 else (1, 2, 32))
    G.set_debug(0)
    G.set_wait_timeout(0)
    G.reduce_scatter(grads, list(shards))
    torch.cuda.synchronize()
    assert G.device_status() == 0
    lay = oracle.plan(g.R, g.rows, g.row_len)
    want = oracle.reduce_scatter(lay, [[t.view(torch.int16).cpu().numpy().view(np.uint16) for t in row]
                                       for row in grads])
    assert np.array_equal(f32_bits(shards), np.stack(want).view(np.uint32))
    G.close()


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_all_gather_matches_oracle(tide, g):
    run_ag(tide, g)  # default: bulk-copy placement for aligned pointers


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_all_gather_register_matches_oracle(tide, g):
    run_ag(tide, g, variant=tide.TIDE_AG_REGISTER)


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_all_gather_bulk_matches_oracle(tide, g):
    run_ag(tide, g, variant=tide.TIDE_AG_BULK)


@pytest.mark.parametrize("ctas", [1, 3, 16, 152])
def test_all_gather_bulk_cta_counts(tide, ctas):
    run_ag(tide, group("qwen3moe").scaled(16), ctas=ctas, variant=tide.TIDE_AG_BULK)
    run_ag(tide, group("llama70b").scaled(16), ctas=ctas, variant=tide.TIDE_AG_BULK)
    run_ag(tide, group("qwen3moe").scaled(16), ctas=ctas, variant=tide.TIDE_AG_BULK, misalign=True)


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_all_gather_ce_matches_oracle(tide, g):
    """1-D copy-engine form: one 1-D copy per (rank, parameter) run of valid rows."""
    copies, uniform = run_ag(tide, g, ce=True, flags=tide.TIDE_FLAG_CE_1D)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    assert not uniform
    assert copies == sum(1 for r in range(g.R) for p in range(g.P) if lay.valid_rows(r, p) > 0)


def _ce_auto_expects_2d(g, lay):
    """The default form rule restated: 2-D when the valid runs average under 4 MiB."""
    runs = sum(1 for r in range(g.R) for p in range(g.P) if lay.valid_rows(r, p) > 0)
    return 2 * lay.U < runs * (4 << 20)


@pytest.mark.parametrize("g", [group("llama70b"), group("qwen3moe").scaled(4), group("tiny")],
                         ids=["llama70b-full", "qwen3moe-div4", "tiny"])
def test_all_gather_ce_default_form(tide, g):
    """No form flag and a uniform pitch: the 2-D form for groups of short runs, the 1-D form for long
    runs (the full Llama-3.1-70B layer); the same rule under TIDE_FLAG_OVERLAP."""
    lay = oracle.plan(g.R, g.rows, g.row_len)
    if lay.U > (1 << 26):  # full-size group: the form choice only, through one unchecked call
        G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
        shards = torch.zeros(g.R, lay.S, dtype=torch.int16, device="cuda")
        params = [torch.empty(g.numel(p), dtype=torch.int16, device="cuda") for p in range(g.P)]
        G.all_gather_ce(list(shards), params)
        torch.cuda.synchronize()
        assert G.last_ce_copies()[1] == int(_ce_auto_expects_2d(g, lay)) == 0
        G.close()
        del shards, params
        torch.cuda.empty_cache()
        return
    copies, uniform = run_ag(tide, g, ce=True)
    assert uniform == _ce_auto_expects_2d(g, lay)
    copies, uniform = run_ag(tide, g, ce=True, flags=tide.TIDE_FLAG_OVERLAP)
    assert uniform == _ce_auto_expects_2d(g, lay)


@pytest.mark.parametrize("g", [group("llama70b").scaled(32), group("qwen3moe").scaled(16), group("tiny")],
                         ids=lambda g: g.name)
def test_overlap_mode_defaults_and_parity(tide, g):
    """TIDE_FLAG_OVERLAP: both SM kernels default to a ninth of the SMs, the copy engines to one lane;
    all three collectives still give the oracle's bits with the defaults."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), tide.TIDE_FLAG_OVERLAP)
    assert G.get_ctas() == (max(1, sms // 9), max(1, sms // 9))
    G.close()
    run_rs(tide, g, flags=tide.TIDE_FLAG_OVERLAP)
    run_ag(tide, g, flags=tide.TIDE_FLAG_OVERLAP)
    copies, uniform = run_ag(tide, g, ce=True, flags=tide.TIDE_FLAG_OVERLAP)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    assert uniform == _ce_auto_expects_2d(g, lay)


@pytest.mark.parametrize("bands", [2, 3, 64])
def test_all_gather_ce_2d_bands_match_oracle(tide, bands):
    """Each parameter's strided copy split into bands of ranks: same bits, min(bands, f_p) 2-D
    copies per parameter plus the partial rank's copy."""
    for g in (group("wan_r16").scaled(8), group("qwen3moe").scaled(16), edge_groups()[1]):
        copies, uniform = run_ag(tide, g, ce=True, flags=tide.TIDE_FLAG_CE_2D, bands=bands)
        assert uniform
        lay = oracle.plan(g.R, g.rows, g.row_len)
        expect = sum(min(bands, r // int(m)) + (r % int(m) > 0) for r, m in zip(g.rows, lay.m))
        assert copies == expect


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_all_gather_ce_2d_matches_oracle(tide, g):
    """The paper's form: one strided (2-D) copy per parameter over its full ranks."""
    copies, uniform = run_ag(tide, g, ce=True, flags=tide.TIDE_FLAG_CE_2D)
    assert uniform
    lay = oracle.plan(g.R, g.rows, g.row_len)
    expect = sum((r // int(m) > 0) + (r % int(m) > 0) for r, m in zip(g.rows, lay.m))
    assert copies == expect


def _shifted_groups():
    """Groups whose small 1-D parameters shift every later prefix offset by 1, 2 or 4 elements, so
    the placement meets every relative alignment of shard and parameter addresses (and a
    Qwen3-shaped group at R = 64, where the per-rank norm pieces of 2 elements do this)."""
    gs = []
    for shift in (1, 2, 3, 4, 5, 7):
        params = []
        for i, (rows, l) in enumerate([(64, 96), (40, 128), (8 * shift, 1), (72, 40), (8 * shift, 1),
                                       (33, 24), (256, 8), (8 * shift + 8, 1), (48, 64)]):
            params.append((f"p{i}", rows, l))
        gs.append(Group(f"shift{shift}", 8, tuple(params)))
    q = group("qwen3moe").scaled(16)
    gs.append(Group("qwen-scaled16-R64", 64, q.params))
    return gs


def test_auto_placement_choice(tide):
    """AUTO resolves to the bulk placement for long runs or a capped CTA count, else the register
    path; explicit choices are kept."""
    long_runs = group("llama70b").scaled(2)  # 72 runs of 2.8 M elements on average
    G = tide.Group(long_runs.R, list(zip(long_runs.rows, long_runs.row_len)))
    assert G.ag_kernel() == tide.TIDE_AG_BULK
    G.set_ctas(0, 16)
    assert G.ag_kernel() == tide.TIDE_AG_BULK
    G.set_ctas(0, 0)
    G.set_ag_variant(tide.TIDE_AG_REGISTER)
    assert G.ag_kernel() == tide.TIDE_AG_REGISTER
    G.set_ag_variant(tide.TIDE_AG_BULK)
    assert G.ag_kernel() == tide.TIDE_AG_BULK
    G.close()
    q = group("qwen3moe").scaled(4)  # 3,144 runs of 12 k elements on average
    G = tide.Group(q.R, list(zip(q.rows, q.row_len)))
    assert G.ag_kernel() == tide.TIDE_AG_REGISTER
    G.set_ctas(0, 16)
    assert G.ag_kernel() == tide.TIDE_AG_BULK
    G.close()


def test_auto_reduce_scatter_choice(tide):
    """AUTO resolves to the TMEM-staged kernel for aligned gradients, at any CTA count and in
    overlap mode; explicit choices are kept."""
    g = group("llama70b").scaled(32)
    for flags in (0, tide.TIDE_FLAG_OVERLAP):
        G = tide.Group(g.R, list(zip(g.rows, g.row_len)), flags)
        assert G.rs_kernel() == tide.TIDE_RS_TMEM
        G.set_ctas(16, 0)
        assert G.rs_kernel() == tide.TIDE_RS_TMEM
        for v in (tide.TIDE_RS_REGISTER, tide.TIDE_RS_BULK, tide.TIDE_RS_TMEM):
            G.set_rs_variant(v)
            assert G.rs_kernel() == v
        G.close()


@pytest.mark.parametrize("variant", [0, 1, 2], ids=["auto", "register", "bulk"])
@pytest.mark.parametrize("g", _shifted_groups(), ids=lambda g: g.name)
def test_all_gather_any_relative_alignment(tide, g, variant):
    run_ag(tide, g, variant=variant)
    run_ag(tide, g, variant=variant, misalign=True)


@pytest.mark.parametrize("g", _shifted_groups(), ids=lambda g: g.name)
def test_reduce_scatter_any_relative_alignment(tide, g):
    run_rs(tide, g)
    run_rs(tide, g, variant=1)


@pytest.mark.parametrize("ctas", [1, 3, 17, 152, 1000])
def test_cta_count_does_not_change_bits(tide, ctas):
    run_rs(tide, group("qwen3moe").scaled(16), ctas=ctas)
    run_ag(tide, group("qwen3moe").scaled(16), ctas=ctas)


def test_misaligned_pointers_take_elementwise_path(tide):
    g = group("llama8b").scaled(32)
    run_rs(tide, g, misalign=True)
    run_ag(tide, g, misalign=True)
    run_ag(tide, g, misalign=True, ce=True)


def test_vec_strict_rejects_misaligned(tide):
    g = group("tiny")
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), tide.TIDE_FLAG_VEC_STRICT)
    grads = [[torch.zeros(g.numel(p) + 1, dtype=torch.bfloat16, device="cuda")[1:] for p in range(g.P)]
             for _ in range(g.R)]
    shards = [torch.zeros(G.S, dtype=torch.float32, device="cuda") for _ in range(g.R)]
    with pytest.raises(tide.TideError) as e:
        G.reduce_scatter(grads, shards)
    assert e.value.status == tide.TIDE_EALIGN


def test_ce_non_uniform_pitch_falls_back(tide):
    g = group("qwen3moe").scaled(16)
    copies, uniform = run_ag(tide, g, ce=True, uniform=False, flags=tide.TIDE_FLAG_CE_2D)
    assert not uniform
    lay = oracle.plan(g.R, g.rows, g.row_len)
    assert copies == sum(1 for r in range(g.R) for p in range(g.P) if lay.valid_rows(r, p) > 0)


def test_ce_strict_rejects_non_uniform_pitch(tide):
    g = group("tiny")
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), tide.TIDE_FLAG_CE_STRICT | tide.TIDE_FLAG_CE_2D)
    buf = torch.zeros(16 * G.S, dtype=torch.bfloat16, device="cuda")
    shards = [buf[a:a + G.S] for a in (0, 2 * G.S, 3 * G.S, 6 * G.S)]  # pitches 2S, S, 3S
    params = [torch.zeros(g.numel(p), dtype=torch.bfloat16, device="cuda") for p in range(g.P)]
    with pytest.raises(tide.TideError) as e:
        G.all_gather_ce(shards, params)
    assert e.value.status == tide.TIDE_ELAYOUT


def test_random_groups(tide):
    for R, rows, row_len in oracle_pins.random_groups(21, 8):
        g = Group(f"random-R{R}", R, tuple((f"p{i}", r, l) for i, (r, l) in enumerate(zip(rows, row_len))))
        run_rs(tide, g)
        run_ag(tide, g)
        run_ag(tide, g, ce=True)


@pytest.mark.parametrize("R", [1024, 4096])
def test_many_ranks(tide, R):
    """Rank counts up to the library's maximum (TIDE_MAX_RANKS): the bulk reduce-scatter's per-piece
    pointer cache grows to 8 R bytes and leaves room for fewer stages; most ranks hold no rows of the
    short parameter, and odd piece offsets mix bulk copies and element-wise sums."""
    g = Group(f"many-ranks-R{R}", R, (("a", 2 * R, 8), ("b", R + R // 2 - 36, 16), ("c", 7, 4)))
    run_rs(tide, g)
    run_rs(tide, g, ctas=16)
    run_ag(tide, g)
    run_ag(tide, g, ce=True)


def test_pointer_table_ring_and_streams(tide):
    """Alternating buffer sets and streams reuse or refill the pointer-table ring correctly."""
    g = group("llama70b").scaled(64)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    sets = []
    for k in range(6):
        gg = Group(g.name, g.R, g.params, grad_seed_per_rank=False, grad_seed=100 + k)
        host = rng.group_grads(gg)
        want = oracle.reduce_scatter(lay, [[t.numpy().view(np.uint16) for t in row] for row in host])
        dev = [[t.cuda() for t in row] for row in host]
        out = [torch.empty(lay.S, dtype=torch.float32, device="cuda") for _ in range(g.R)]
        sets.append((dev, out, want))
    streams = [torch.cuda.Stream() for _ in range(2)]
    for it in range(3):
        for k, (dev, out, want) in enumerate(sets):
            st = streams[(k + it) % 2]
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                for o in out:
                    o.fill_(float("nan"))
                G.reduce_scatter(dev, out)
            torch.cuda.synchronize()
            for d in range(g.R):
                assert np.array_equal(f32_bits(out[d]), want[d].view(np.uint32)), (it, k, d)
    G.close()


def test_premarshalled_pointer_tables(tide):
    """Pointer tables marshalled once with pointer_table give the same bits as tensor lists, for
    the reduce-scatter and both placements, on a many-parameter group."""
    g = group("qwen3moe").scaled(16)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    host = rng.group_grads(g)
    want = oracle.reduce_scatter(lay, [[t.numpy().view(np.uint16) for t in row] for row in host])
    dev = [[t.cuda() for t in row] for row in host]
    out = [torch.full((lay.S,), float("nan"), device="cuda") for _ in range(g.R)]
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    gt = tide.pointer_table([t for row in dev for t in row])
    st = tide.pointer_table(out)
    for _ in range(2):
        G.reduce_scatter(gt, st)
    torch.cuda.synchronize()
    for d in range(g.R):
        assert np.array_equal(f32_bits(out[d]), want[d].view(np.uint32)), d
    shards = [rng.shard_bits(g, r, lay.S).cuda() for r in range(g.R)]
    ref = [torch.empty(g.numel(p), dtype=torch.int16, device="cuda") for p in range(g.P)]
    G.all_gather(shards, ref)
    for ce in (False, True):
        got = [torch.zeros(g.numel(p), dtype=torch.int16, device="cuda") for p in range(g.P)]
        (G.all_gather_ce if ce else G.all_gather)(tide.pointer_table(shards), tide.pointer_table(got))
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, ref)), ce
    G.close()


# ---- full sizes, launch configuration of the benchmark ---------------------------------------

FULL = ["llama8b", "qwen3moe", "llama70b", "wan_r8", "wan_r16", "wan_r32", "wan_r64"]


def _sample_positions(lay, seed, n=3000):
    """Random shard positions plus the first/last element of every piece and both sides of
    every valid/padding boundary."""
    rs = np.random.default_rng(seed)
    d = list(rs.integers(0, lay.R, n))
    j = list(rs.integers(0, lay.S, n))
    for dd in range(lay.R):
        for p in range(lay.P):
            o, s = int(lay.o[p]), int(lay.s[p])
            v = lay.valid_rows(dd, p) * int(lay.row_len[p])
            for x in {o, o + s - 1, o + v - 1, o + v}:
                if o <= x < o + s:
                    d.append(dd)
                    j.append(x)
    return np.asarray(d, np.int64), np.asarray(j, np.int64)


FULL_CASES = [(n, 0, 0) for n in FULL] + [("llama70b", 16, 0), ("qwen3moe", 16, 0), ("wan_r64", 24, 0),
                                          ("llama70b", 0, 3), ("llama70b", 16, 3), ("qwen3moe", 16, 3)]


@pytest.mark.parametrize("name,ctas,variant", FULL_CASES,
                         ids=[f"{n}-ctas{c or 'default'}{'-tmem' if v == 3 else ''}" for n, c, v in FULL_CASES])
def test_full_size_reduce_scatter(tide, name, ctas, variant):
    """Default CTAs = the benchmark's step; capped CTAs = the automatic bulk-copy path the
    interference harness times; variant 3 = the TMEM-staged kernel."""
    g = group(name)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    grads = [[rng.grad_bits(g, r, p, device="cuda").view(torch.bfloat16) for p in range(g.P)] for r in range(g.R)]
    shards = torch.empty(g.R, lay.S, dtype=torch.float32, device="cuda")
    shards.view(torch.int32).fill_(F32_SENTINEL)
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    G.set_ctas(ctas, 0)
    G.set_rs_variant(variant)
    G.reduce_scatter(grads, list(shards))
    torch.cuda.synchronize()
    assert G.device_status() == 0
    # (1) sampled outputs, computed one by one by the oracle from regenerated inputs
    d, j = _sample_positions(lay, seed=len(name))
    want = oracle.rs_points(lay, d, j, lambda r, p, idx: rng.grad_bits(g, r, p, idx=torch.from_numpy(idx))
                            .numpy().view(np.uint16))
    got = shards[torch.from_numpy(d).cuda(), torch.from_numpy(j).cuda()]
    assert np.array_equal(f32_bits(got), want.view(np.uint32))
    # (2) every element written; every padding element +0.0; every piece equal to torch fp32 adds in
    # ascending rank order (the definition, evaluated with torch on the device)
    assert not bool((shards.view(torch.int32) == F32_SENTINEL).any())
    for dd in range(g.R):
        for p in range(g.P):
            o, s, L = int(lay.o[p]), int(lay.s[p]), int(lay.row_len[p])
            v = lay.valid_rows(dd, p) * L
            piece = shards[dd, o:o + s]
            assert bool((piece[v:].view(torch.int32) == 0).all())
            if v:
                acc = grads[0][p][dd * s: dd * s + v].float()
                for r in range(1, g.R):
                    acc = acc + grads[r][p][dd * s: dd * s + v].float()
                assert torch.equal(piece[:v].view(torch.int32), acc.view(torch.int32)), (dd, p)
    # (3) total over all shards = total gradient (fp64), within the fp32 fold bound
    tot_in = sum(grads[r][p].double().sum() for r in range(g.R) for p in range(g.P)).item()
    abs_in = sum(grads[r][p].double().abs().sum() for r in range(g.R) for p in range(g.P)).item()
    tot_out = shards.double().sum().item()
    assert abs(tot_out - tot_in) <= (g.R - 1) * 2.0 ** -24 * abs_in
    G.close()
    del grads, shards
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", FULL)
def test_full_size_all_gather(tide, name):
    g = group(name)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    shards = torch.stack([rng.shard_bits(g, r, lay.S, device="cuda") for r in range(g.R)])
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    for mode in ("register", "ce", "bulk"):
        ce = mode == "ce"
        G.set_ag_variant(tide.TIDE_AG_BULK if mode == "bulk" else tide.TIDE_AG_REGISTER)
        params = [torch.full((g.numel(p),), BF16_SENTINEL, dtype=torch.int16, device="cuda") for p in range(g.P)]
        (G.all_gather_ce if ce else G.all_gather)(list(shards), params)
        torch.cuda.synchronize()
        assert G.device_status() == 0
        rs = np.random.default_rng(7)
        for p in range(g.P):
            n = g.numel(p)
            idx = np.unique(np.concatenate([rs.integers(0, n, 64), [0, n - 1]]))
            r, jj = oracle.ag_points(lay, p, idx)
            want = np.zeros(idx.size, np.int64)
            for a in np.unique(r):
                sel = r == a
                want[sel] = rng.shard_bits(g, int(a), 0, idx=torch.from_numpy(jj[sel])).numpy().astype(np.int64)
            want &= 0xFFFF
            got = params[p][torch.from_numpy(idx).cuda()].cpu().numpy().astype(np.int64) & 0xFFFF
            assert np.array_equal(got, want), (mode, p)
            for rr in range(g.R):
                v = lay.valid_rows(rr, p) * int(lay.row_len[p])
                s, o = int(lay.s[p]), int(lay.o[p])
                assert torch.equal(params[p][rr * s: rr * s + v], shards[rr, o:o + v]), (mode, p, rr)
        del params
    G.close()
    del shards
    torch.cuda.empty_cache()


@pytest.mark.parametrize("g", [group("tiny"), group("llama70b").scaled(32), group("qwen3moe").scaled(16),
                               group("wan_r64").scaled(16)], ids=lambda g: g.name)
def test_slot_reuse_staging(tide, g):
    """Gradients staged into all-gather-sized slots, the originals overwritten right after (as if
    released), then the reduce-scatter from the slots: the oracle's result, bit for bit."""
    lay = oracle.plan(g.R, g.rows, g.row_len)
    host = rng.group_grads(g)
    want = np.stack(oracle.reduce_scatter(lay, [[t.numpy().view(np.uint16) for t in row] for row in host]))
    grads = [[t.cuda() for t in row] for row in host]
    slot_elems = g.R * lay.S
    slots = torch.full((g.R, slot_elems), BF16_SENTINEL, dtype=torch.int16, device="cuda")
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    staged = G.stage_into_slots(grads, list(slots), slot_elems)
    for row in grads:  # released: later work reuses the memory (here: overwritten with NaN bits)
        for t in row:
            t.fill_(0x7FC0)
    out = torch.empty(g.R, lay.S, dtype=torch.float32, device="cuda")
    G.reduce_scatter(staged, list(out))
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(out), want.view(np.uint32))
    # the slots hold each rank's unsharded gradients packed in parameter order
    flat = slots.cpu().numpy().view(np.uint16)
    for r in range(g.R):
        packed = np.concatenate([host[r][p].numpy().view(np.uint16) for p in range(g.P)])
        assert np.array_equal(flat[r, :packed.size], packed)
        assert np.all(flat[r, packed.size:] == (BF16_SENTINEL & 0xFFFF))
    with pytest.raises(tide.TideError) as e:
        G.stage_into_slots(grads, list(slots), lay.U - 1)
    assert e.value.status == tide.TIDE_ERANGE
    G.close()


@pytest.mark.parametrize("lanes", [1, 2, 4, 8])
@pytest.mark.parametrize("flags", [0, 4], ids=["1d", "2d"])
def test_ce_lanes_stay_stream_ordered(tide, lanes, flags):
    """Copy-engine placement spread over helper streams: it sees work enqueued just before it on the
    caller's stream and the caller's stream sees its result right after, with no host sync."""
    g = group("qwen3moe").scaled(8)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    src = torch.stack([rng.shard_bits(g, r, lay.S) for r in range(g.R)]).cuda()
    want = oracle.all_gather(lay, [a.cpu().numpy().view(np.uint16) for a in src],
                             [np.zeros(g.numel(p), np.uint16) for p in range(g.P)])
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), flags)
    G.set_ce_lanes(lanes)
    st = torch.cuda.Stream()
    shards = torch.zeros_like(src)
    params = [torch.zeros(g.numel(p), dtype=torch.int16, device="cuda") for p in range(g.P)]
    outs = [torch.empty_like(x) for x in params]
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        torch.cuda._sleep(2_000_000)  # keep the stream busy so ordering, not luck, decides
        shards.copy_(src)
        G.all_gather_ce(list(shards), params, st)
        for o, x in zip(outs, params):
            o.copy_(x)
    torch.cuda.synchronize()
    for p in range(g.P):
        assert np.array_equal(outs[p].cpu().numpy().view(np.uint16), want[p]), (lanes, p)
    G.close()


def test_element_misaligned_pointers_are_rejected(tide):
    """Pointers that are not aligned to their element size are refused before anything runs."""
    g = group("tiny")
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    raw = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
    odd = raw.data_ptr() + 1   # not 2-byte aligned
    two = raw.data_ptr() + 2   # 2-byte but not 4-byte aligned
    good16 = raw.data_ptr()
    grads = [[good16] * g.P for _ in range(g.R)]
    for bad_g, bad_s in ((odd, good16), (good16, two)):
        gp = [[bad_g if (r, p) == (1, 1) else good16 for p in range(g.P)] for r in range(g.R)]
        sp = [bad_s if d == 2 else good16 for d in range(g.R)]
        with pytest.raises(tide.TideError) as e:
            G.reduce_scatter(gp, sp)
        assert e.value.status == tide.TIDE_EINVAL
    with pytest.raises(tide.TideError) as e:
        G.all_gather([good16] * g.R, [odd] + [good16] * (g.P - 1))
    assert e.value.status == tide.TIDE_EINVAL
    torch.cuda.synchronize()
    G.close()


def test_shards_need_only_fp32_alignment(tide):
    """Shard pointers 4 or 8 bytes past a 16-byte boundary keep the vector paths (same bits)."""
    g = group("llama8b").scaled(32)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    host = rng.group_grads(g)
    want = oracle.reduce_scatter(lay, [[t.numpy().view(np.uint16) for t in row] for row in host])
    grads = [[t.cuda() for t in row] for row in host]
    for off in (1, 2, 3):
        buf = torch.full((g.R, lay.S + 4), float("nan"), device="cuda")
        shards = [buf[d, off:off + lay.S] for d in range(g.R)]
        for variant in (tide.TIDE_RS_BULK, tide.TIDE_RS_REGISTER):
            G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
            G.set_rs_variant(variant)
            G.reduce_scatter(grads, shards)
            torch.cuda.synchronize()
            for d in range(g.R):
                assert np.array_equal(f32_bits(shards[d]), want[d].view(np.uint32)), (off, variant, d)
            G.close()


# ---- the summing step over staging slots (the reduce-scatter's local step on R GPUs) -----------


def fill_slots(g, lay, grads, d, slots):
    """Destination d's exchange, with device copies standing in for the copies from the other
    GPUs: from every contributor r, its slice d of every parameter into slot r at o_p."""
    from all_gather_tide_gb300 import exchange

    for c in exchange.reduce_scatter_pulls(g.R, g.rows, g.row_len, d):
        slots[c.src_rank][c.dst_off:c.dst_off + c.elems].copy_(grads[c.src_rank][c.param][c.src_off:c.src_off + c.elems])


def run_rs_slots(tide, g, dests=None, ctas=0, misalign=False, flags=0, library_staging=False, lanes=0, variant=0):
    lay = oracle.plan(g.R, g.rows, g.row_len)
    host = rng.group_grads(g)
    want = oracle.reduce_scatter(lay, [[t.numpy().view(np.uint16) for t in row] for row in host])
    grads = [[t.cuda().view(-1) for t in row] for row in host]
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), flags)
    G.set_ctas(ctas, 0)
    G.set_rs_variant(variant)
    if lanes:
        G.set_ce_lanes(lanes)
    off = 1 if misalign else 0
    for d in (range(g.R) if dests is None else dests):
        packed = Guarded(g.R * lay.S, torch.int16, fill=BF16_JUNK, offset_elems=off)  # junk in the padding
        slots = [packed.view[r * lay.S:(r + 1) * lay.S] for r in range(g.R)]
        if library_staging:
            G.stage_slices(d, grads, slots)  # copy engines, on the same stream as the sum
        else:
            fill_slots(g, lay, grads, d, slots)
        shard = Guarded(lay.S, torch.float32, fill=F32_SENTINEL)
        G.reduce_scatter_slots(d, slots, shard.view)
        torch.cuda.synchronize()
        assert G.device_status() == 0
        got = f32_bits(shard.view)
        bad = np.nonzero(got != want[d].view(np.uint32))[0]
        assert bad.size == 0, f"{g.name}: shard {d} from slots differs at {bad[:8]} (of {bad.size})"
        assert shard.guards_intact() and packed.guards_intact(), f"{g.name}: guard band overwritten ({d})"
    G.close()


def _slot_dests(g):
    return None if g.R <= 16 else sorted({0, 1, g.R // 2, g.R - 1})


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_reduce_scatter_slots_matches_oracle(tide, g):
    run_rs_slots(tide, g, _slot_dests(g))


@pytest.mark.parametrize("g", [group("tiny"), group("llama70b").scaled(32), edge_groups()[2], edge_groups()[3]],
                         ids=lambda g: g.name)
def test_reduce_scatter_slots_misaligned_slots(tide, g):
    """Slots that are only 2-byte aligned take the element-wise path: same bits."""
    run_rs_slots(tide, g, _slot_dests(g), misalign=True)


@pytest.mark.parametrize("g", reduced_groups(), ids=_ids(reduced_groups()))
def test_stage_slices_then_sum_matches_oracle(tide, g):
    """The library's own exchange copies (tide_stage_slices) followed by the summing step."""
    run_rs_slots(tide, g, _slot_dests(g), library_staging=True)


@pytest.mark.parametrize("lanes", [1, 3, 8])
def test_stage_slices_lanes_stay_stream_ordered(tide, lanes):
    run_rs_slots(tide, group("qwen3moe").scaled(16), [0, 3, 7], library_staging=True, lanes=lanes)
    run_rs_slots(tide, edge_groups()[2], None, library_staging=True, lanes=lanes, misalign=True)


@pytest.mark.parametrize("g", [group("tiny"), group("llama70b").scaled(32), group("wan_r64").scaled(16)],
                         ids=lambda g: g.name)
def test_reduce_scatter_slots_tmem(tide, g):
    run_rs_slots(tide, g, _slot_dests(g), variant=tide.TIDE_RS_TMEM)
    run_rs_slots(tide, g, _slot_dests(g), ctas=16, variant=tide.TIDE_RS_TMEM)


@pytest.mark.parametrize("ctas", [1, 3, 16, 1000])
def test_reduce_scatter_slots_cta_counts(tide, ctas):
    run_rs_slots(tide, group("qwen3moe").scaled(16), [0, 5, 7], ctas=ctas)


def test_reduce_scatter_slots_rejects_bad_arguments(tide):
    g = group("tiny")
    lay = oracle.plan(g.R, g.rows, g.row_len)
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)), tide.TIDE_FLAG_VEC_STRICT)
    slots = torch.zeros(g.R, lay.S + 8, dtype=torch.int16, device="cuda")
    shard = torch.zeros(lay.S + 1, dtype=torch.float32, device="cuda")
    good = [slots[r, :lay.S] for r in range(g.R)]
    for d in (-1, g.R):
        with pytest.raises(tide.TideError) as e:
            G.reduce_scatter_slots(d, good, shard)
        assert e.value.status == tide.TIDE_EINVAL
    odd = torch.zeros(lay.S + 1, dtype=torch.float32, device="cuda").view(torch.int16)[1:]  # 2-byte aligned only
    with pytest.raises(tide.TideError) as e:
        G.reduce_scatter_slots(0, good, odd)  # an fp32 shard needs 4-byte alignment
    assert e.value.status == tide.TIDE_EINVAL
    with pytest.raises(tide.TideError) as e:
        G.reduce_scatter_slots(0, [slots[r, 1:lay.S + 1] for r in range(g.R)], shard)
    assert e.value.status == tide.TIDE_EALIGN  # VEC_STRICT: slots not 16-byte aligned
    G.close()


@pytest.mark.parametrize("name", ["llama70b", "wan_r64"])
def test_full_size_reduce_scatter_slots(tide, name):
    """Full-size groups at the default grid, first and last destination: sampled outputs computed
    one by one by the oracle, and every piece equal to torch fp32 adds in ascending rank order."""
    g = group(name)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    grads = [[rng.grad_bits(g, r, p, device="cuda").view(-1) for p in range(g.P)] for r in range(g.R)]
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    slots = torch.empty(g.R, lay.S, dtype=torch.int16, device="cuda")
    shard = torch.empty(lay.S, dtype=torch.float32, device="cuda")
    dd_all, jj_all = _sample_positions(lay, seed=7 + len(name))
    for d in (0, g.R - 1):
        slots.fill_(BF16_JUNK)
        shard.view(torch.int32).fill_(F32_SENTINEL)
        fill_slots(g, lay, grads, d, list(slots))
        G.reduce_scatter_slots(d, list(slots), shard)
        torch.cuda.synchronize()
        assert G.device_status() == 0
        j = jj_all[dd_all == d]
        want = oracle.rs_points(lay, np.full(j.shape, d, np.int64), j,
                                lambda r, p, idx: rng.grad_bits(g, r, p, idx=torch.from_numpy(idx)).numpy().view(np.uint16))
        got = shard[torch.from_numpy(j).cuda()]
        assert np.array_equal(f32_bits(got), want.view(np.uint32)), d
        for p in range(g.P):
            o, s, L = int(lay.o[p]), int(lay.s[p]), int(lay.row_len[p])
            v = lay.valid_rows(d, p) * L
            piece = shard[o:o + s]
            assert bool((piece[v:].view(torch.int32) == 0).all()), (d, p)
            if v:
                acc = grads[0][p][d * s: d * s + v].view(torch.bfloat16).float()
                for r in range(1, g.R):
                    acc = acc + grads[r][p][d * s: d * s + v].view(torch.bfloat16).float()
                assert torch.equal(piece[:v].view(torch.int32), acc.view(torch.int32)), (d, p)
    G.close()
    del grads, slots, shard
    torch.cuda.empty_cache()

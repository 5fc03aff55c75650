"""The C ABI library on the CPU: it builds, loads, exports every declared symbol, its host-only
planner matches the oracle's on every workload, and argument checks fail before any CUDA call."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

import oracle
from workloads import GROUPS, group

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tide():
    from all_gather_tide_gb300 import build

    build.build()
    import all_gather_tide_gb300 as t

    t.lib()
    return t


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "tide.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tide_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(tide):
    names = _declared_symbols()
    assert len(names) >= 16
    L = tide.lib()
    for n in names:
        assert hasattr(L, n), n
        assert n in tide.SIGNATURES, n
    assert set(tide.SIGNATURES) == set(names)


def test_version_and_strerror(tide):
    assert tide.tide_version() == 100
    for st in range(0, -7, -1):
        assert tide.tide_strerror(st) and tide.tide_strerror(st) != "unknown status"
    assert tide.tide_strerror(-99) == "unknown status"


@pytest.mark.parametrize("name", sorted(GROUPS))
def test_planner_matches_oracle(tide, name):
    g = group(name)
    m, s, o, S, U = tide.tide_plan_layout(g.R, g.rows, g.row_len)
    lay = oracle.plan(g.R, g.rows, g.row_len)
    assert m == lay.m.tolist() and s == lay.s.tolist() and o == lay.o.tolist()
    assert (S, U) == (lay.S, lay.U)


def test_planner_matches_oracle_random(tide):
    import oracle_pins

    for R, rows, row_len in oracle_pins.random_groups(11, 50):
        m, s, o, S, U = tide.tide_plan_layout(R, rows, row_len)
        lay = oracle.plan(R, rows, row_len)
        assert m == lay.m.tolist() and s == lay.s.tolist() and o == lay.o.tolist() and (S, U) == (lay.S, lay.U)


def _create_status(tide, R, rows, row_len, flags=0, out=True):
    L = tide.lib()
    h = ctypes.c_void_p()
    arr = lambda xs: (ctypes.c_int64 * max(1, len(xs)))(*xs)
    return L.tide_group_create(ctypes.byref(h) if out else None, R, len(rows), arr(rows), arr(row_len), flags)


def test_create_rejects_bad_arguments_before_cuda(tide):
    assert _create_status(tide, 0, [4], [4]) == tide.TIDE_EINVAL
    assert _create_status(tide, 5000, [4], [4]) == tide.TIDE_EINVAL
    assert _create_status(tide, 2, [0], [4]) == tide.TIDE_EINVAL
    assert _create_status(tide, 2, [4], [-1]) == tide.TIDE_EINVAL
    assert _create_status(tide, 2, [], []) == tide.TIDE_EINVAL
    assert _create_status(tide, 2, [4], [4], out=False) == tide.TIDE_EINVAL
    assert _create_status(tide, 2, [1 << 40], [1 << 30]) == tide.TIDE_ERANGE
    # unknown flags and contradictory copy-engine forms
    assert _create_status(tide, 2, [4], [4], flags=0x100) == tide.TIDE_EINVAL
    assert _create_status(tide, 2, [4], [4], flags=tide.TIDE_FLAG_CE_1D | tide.TIDE_FLAG_CE_2D) == tide.TIDE_EINVAL
    assert _create_status(tide, 2, [4], [4], flags=tide.TIDE_FLAG_CE_1D | tide.TIDE_FLAG_CE_STRICT) == tide.TIDE_EINVAL


def test_plan_layout_rejects(tide):
    with pytest.raises(tide.TideError) as e:
        tide.tide_plan_layout(0, [1], [1])
    assert e.value.status == tide.TIDE_EINVAL
    with pytest.raises(tide.TideError) as e:
        tide.tide_plan_layout(8, [1 << 62], [4])
    assert e.value.status == tide.TIDE_ERANGE


def test_null_group_calls(tide):
    L = tide.lib()
    arr = (ctypes.c_void_p * 1)(0)
    for fn in ("tide_reduce_scatter", "tide_all_gather", "tide_all_gather_ce"):
        assert getattr(L, fn)(None, arr, arr, None) == tide.TIDE_EINVAL
    v = ctypes.c_int64()
    assert L.tide_group_shard_elems(None, ctypes.byref(v)) == tide.TIDE_EINVAL
    k = ctypes.c_int32()
    assert L.tide_group_ag_kernel(None, ctypes.byref(k)) == tide.TIDE_EINVAL
    assert L.tide_group_rs_kernel(None, ctypes.byref(k)) == tide.TIDE_EINVAL
    assert L.tide_group_set_ce_bands(None, 2) == tide.TIDE_EINVAL
    assert L.tide_reduce_scatter_slots(None, 0, arr, 16, None) == tide.TIDE_EINVAL
    assert L.tide_stage_slices(None, 0, arr, arr, None) == tide.TIDE_EINVAL
    assert L.tide_group_destroy(None) == tide.TIDE_OK


def test_probe_argument_checks_before_cuda(tide):
    L = tide.lib()
    assert L.tide_probe_hold(0, 128, 0, 1, 1000, None, None) == tide.TIDE_EINVAL
    assert L.tide_probe_hold(6, 128, 0, 4, 1000, None, None) == tide.TIDE_EINVAL  # not whole clusters
    assert L.tide_probe_hold(4, 2048, 0, 1, 1000, None, None) == tide.TIDE_EINVAL
    assert L.tide_probe_bulk_read(None, 1024, 1, 4096, 4, None, None) == tide.TIDE_EINVAL
    assert L.tide_probe_bulk_read(16, 1024, 1, 4095, 4, 16, None) == tide.TIDE_EINVAL
    assert L.tide_probe_bulk_read(16, 1024, 1, 65536, 4, 16, None) == tide.TIDE_EINVAL  # > 200 KB staged
    ok = dict(buf=256, bulk=1 << 20, ldg=1 << 20, ctas=16, copy=46080, stages=4, cons=8, ldgw=7, out=16)
    for k, bad in (("buf", 0), ("buf", 272), ("ctas", 0), ("copy", 46081), ("stages", 17), ("stages", 6),
                   ("cons", -1), ("ldgw", 8), ("ldg", 33), ("out", 0)):
        args = dict(ok, **{k: bad})
        assert L.tide_probe_ingest(*args.values(), None) == tide.TIDE_EINVAL, (k, bad)
    ok = dict(buf=256, bulk=1 << 20, st=512, stb=1 << 20, ctas=16, copy=73728, stages=3, cons=11, stw=4, br=8, bv=6,
              out=16)
    for k, bad in (("buf", 0), ("buf", 272), ("st", 0), ("st", 528), ("stb", 33), ("ctas", 0), ("copy", 46081),
                   ("stages", 4), ("cons", 0), ("stw", 5), ("stw", -1), ("br", -1), ("bv", -1), ("stb", 32 * 15),
                   ("out", 0)):
        args = dict(ok, **{k: bad})
        assert L.tide_probe_mixed(*args.values(), None) == tide.TIDE_EINVAL, (k, bad)


def test_pointer_table_marshalling(tide):
    import torch

    xs = [torch.empty(3, dtype=torch.int16) for _ in range(5)] + [12345]
    t = tide.pointer_table(xs)
    assert [v for v in t] == [x.data_ptr() for x in xs[:5]] + [12345]
    assert tide._ptr_array(t) is t and tide._flat_grads(t) is t
    L = tide.lib()
    assert L.tide_reduce_scatter(None, t, t, None) == tide.TIDE_EINVAL


def test_header_constants_match_binding(tide):
    """Every integer constant the header defines has the same value in the binding (where the binding
    exposes it)."""
    src = open(os.path.join(ROOT, "include", "tide.h")).read()
    seen = 0
    for name, value in re.findall(r"^#define\s+(TIDE_\w+)\s+([^/\n]+)", src, flags=re.M):
        expr = value.strip().replace("u", "")
        if not re.fullmatch(r"[-()0-9x<\s]+", expr):
            continue
        v = eval(expr)  # integer literals, shifts and parentheses only
        if hasattr(tide, name):
            assert getattr(tide, name) == v, name
            seen += 1
    assert seen >= 15


def test_missing_library_fails_loudly(tmp_path):
    """Without libtide.so the binding raises on first use: there is no fallback path."""
    code = (
        "import all_gather_tide_gb300 as t\n"
        f"t.LIB_PATH = {str(tmp_path / 'libtide.so')!r}\n"
        "t._lib = None\n"
        "try:\n"
        "    t.Group(2, [(4, 3)])\n"
        "except RuntimeError as e:\n"
        "    assert 'missing' in str(e), e\n"
        "    print('raised')\n"
    )
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == "raised", out.stdout + out.stderr

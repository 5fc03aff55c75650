"""CPU oracle of the TIDE reduce-scatter / all-gather placement (TEST INFRASTRUCTURE ONLY).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this package.
It wraps ``tide_oracle.c`` (plain C loops, built with gcc) with numpy marshalling, and adds one
numpy routine that evaluates single reduce-scatter outputs from their inputs, for checking
sampled outputs of full-size GPU runs.  It shares no code with the CUDA library and never
imports it.

"TIDE" is "The Endgame of FSDP Communication: Layout-Aware Collectives on Copy Engines, RDMA,
and NVSwitch" (arXiv 2610.38228); the definitions followed are cited in ``tide_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Callable, List, NamedTuple, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tide_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]

_i64p = ctypes.POINTER(ctypes.c_int64)
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library with gcc (no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _configure(L: ctypes.CDLL) -> ctypes.CDLL:
    i32 = ctypes.c_int32
    vpp = ctypes.POINTER(ctypes.c_void_p)
    L.oracle_plan.argtypes = [i32, i32, _i64p, _i64p, _i64p, _i64p, _i64p, _i64p, _i64p]
    L.oracle_valid_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, i32]
    L.oracle_valid_rows.restype = ctypes.c_int64
    L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f32.restype = ctypes.c_float
    for fn in ("oracle_reduce_scatter", "oracle_exact_sum", "oracle_all_gather", "oracle_shard_bf16"):
        getattr(L, fn).argtypes = [i32, i32, _i64p, _i64p, vpp, vpp]
    for fn in ("oracle_reduce_scatter_part", "oracle_all_gather_part"):
        getattr(L, fn).argtypes = [i32, i32, _i64p, _i64p, vpp, vpp, i32, i32, i32]
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


def use_library(path: str):
    """Point this module at another build of ``tide_oracle.c`` (tests use it to run the pins
    against deliberately broken copies of the oracle); returns the previous library."""
    global _lib
    prev = _lib
    _lib = _configure(ctypes.CDLL(path)) if path else None
    return prev


def restore_library(prev) -> None:
    global _lib
    _lib = prev


def _i64(a: Sequence[int]) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _ptrs(arrs: Sequence[np.ndarray]):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


class Layout(NamedTuple):
    R: int
    rows: np.ndarray
    row_len: np.ndarray
    m: np.ndarray  # padded per-rank rows of each parameter
    s: np.ndarray  # per-rank shard elements of each parameter
    o: np.ndarray  # prefix offset (elements) of each parameter in a rank's packed shard
    S: int  # per-rank packed shard elements
    U: int  # unsharded group elements

    @property
    def P(self) -> int:
        return len(self.rows)

    def valid_rows(self, d: int, p: int) -> int:
        return int(lib().oracle_valid_rows(int(self.rows[p]), int(self.m[p]), d))


def plan(R: int, rows: Sequence[int], row_len: Sequence[int]) -> Layout:
    """Table 2 quantities of a group: m_p, s_p, o_p, S, U."""
    rows_a, len_a = _i64(rows), _i64(row_len)
    P = len(rows_a)
    m, s, o = (np.zeros(P, np.int64) for _ in range(3))
    S, U = ctypes.c_int64(), ctypes.c_int64()
    rc = lib().oracle_plan(R, P, rows_a.ctypes.data_as(_i64p), len_a.ctypes.data_as(_i64p),
                           m.ctypes.data_as(_i64p), s.ctypes.data_as(_i64p), o.ctypes.data_as(_i64p),
                           ctypes.byref(S), ctypes.byref(U))
    if rc != 0:
        raise ValueError(f"oracle_plan rejected the group (rc={rc})")
    return Layout(R, rows_a, len_a, m, s, o, S.value, U.value)


def _check_grads(lay: Layout, grads):
    assert len(grads) == lay.R and all(len(g) == lay.P for g in grads)
    flat = []
    for r in range(lay.R):
        for p in range(lay.P):
            a = np.ascontiguousarray(grads[r][p]).view(np.uint16).reshape(-1)
            assert a.size == lay.rows[p] * lay.row_len[p]
            flat.append(a)
    return flat


def reduce_scatter(lay: Layout, grads: Sequence[Sequence[np.ndarray]]) -> List[np.ndarray]:
    """``grads[r][p]`` (bf16 bits, uint16/int16, flat) -> R fp32 shards of S elements."""
    flat = _check_grads(lay, grads)
    shards = [np.empty(lay.S, np.float32) for _ in range(lay.R)]
    rc = lib().oracle_reduce_scatter(lay.R, lay.P, lay.rows.ctypes.data_as(_i64p),
                                     lay.row_len.ctypes.data_as(_i64p), _ptrs(flat), _ptrs(shards))
    assert rc == 0
    return shards


class Marshalled(NamedTuple):
    """Pointer tables of one group's host arrays, built once so that many part calls (possibly
    from several threads; ctypes releases the GIL during each call) reuse them."""
    lay: Layout
    src: object
    dst: object
    keep: tuple  # the arrays the tables point into


def marshal_reduce_scatter(lay: Layout, grads, shards: Sequence[np.ndarray]) -> Marshalled:
    """Pointer tables for ``reduce_scatter_part``: ``grads[r][p]`` bf16 bits, ``shards`` R fp32
    arrays of S elements (written in place)."""
    flat = _check_grads(lay, grads)
    assert len(shards) == lay.R and all(s.dtype == np.float32 and s.size >= lay.S for s in shards)
    return Marshalled(lay, _ptrs(flat), _ptrs(shards), (flat, list(shards)))


def reduce_scatter_part(m: Marshalled, d: int, p_begin: int, p_end: int) -> None:
    """Destination rank ``d``'s shard elements of parameters ``p_begin <= p < p_end`` only."""
    lay = m.lay
    rc = lib().oracle_reduce_scatter_part(lay.R, lay.P, lay.rows.ctypes.data_as(_i64p),
                                          lay.row_len.ctypes.data_as(_i64p), m.src, m.dst, d, p_begin, p_end)
    assert rc == 0, rc


def marshal_all_gather(lay: Layout, shards: Sequence[np.ndarray], params: Sequence[np.ndarray]) -> Marshalled:
    """Pointer tables for ``all_gather_part``: R bf16 shards, P bf16 parameters (written in place)."""
    sh = [np.ascontiguousarray(s).view(np.uint16).reshape(-1) for s in shards]
    assert len(sh) == lay.R and all(s.size >= lay.S for s in sh)
    pa = [p.view(np.uint16).reshape(-1) for p in params]
    assert len(pa) == lay.P and all(pa[p].size == lay.rows[p] * lay.row_len[p] for p in range(lay.P))
    return Marshalled(lay, _ptrs(sh), _ptrs(pa), (sh, pa))


def all_gather_part(m: Marshalled, r: int, p_begin: int, p_end: int) -> None:
    """Source rank ``r``'s rows of parameters ``p_begin <= p < p_end`` only."""
    lay = m.lay
    rc = lib().oracle_all_gather_part(lay.R, lay.P, lay.rows.ctypes.data_as(_i64p),
                                      lay.row_len.ctypes.data_as(_i64p), m.src, m.dst, r, p_begin, p_end)
    assert rc == 0, rc


def exact_sum(lay: Layout, grads) -> List[np.ndarray]:
    """Same layout as ``reduce_scatter`` with the sums taken in fp64."""
    flat = _check_grads(lay, grads)
    out = [np.empty(lay.S, np.float64) for _ in range(lay.R)]
    rc = lib().oracle_exact_sum(lay.R, lay.P, lay.rows.ctypes.data_as(_i64p),
                                lay.row_len.ctypes.data_as(_i64p), _ptrs(flat), _ptrs(out))
    assert rc == 0
    return out


def all_gather(lay: Layout, shards: Sequence[np.ndarray], params: Sequence[np.ndarray]) -> List[np.ndarray]:
    """Place R packed bf16 shards into per-parameter tensors (``params`` are written in place
    and returned, so a caller can prefill them with a sentinel)."""
    sh = [np.ascontiguousarray(s).view(np.uint16).reshape(-1) for s in shards]
    assert len(sh) == lay.R and all(s.size >= lay.S for s in sh)
    pa = [p.view(np.uint16).reshape(-1) for p in params]
    assert len(pa) == lay.P and all(pa[p].size == lay.rows[p] * lay.row_len[p] for p in range(lay.P))
    rc = lib().oracle_all_gather(lay.R, lay.P, lay.rows.ctypes.data_as(_i64p),
                                 lay.row_len.ctypes.data_as(_i64p), _ptrs(sh), _ptrs(pa))
    assert rc == 0
    return list(params)


def shard_bf16(lay: Layout, params: Sequence[np.ndarray], shards: Sequence[np.ndarray]) -> List[np.ndarray]:
    """Pack per-parameter bf16 tensors into R shards; padding positions keep their prior content."""
    pa = [np.ascontiguousarray(p).view(np.uint16).reshape(-1) for p in params]
    sh = [s.view(np.uint16).reshape(-1) for s in shards]
    assert len(sh) == lay.R and all(s.size >= lay.S for s in sh)
    rc = lib().oracle_shard_bf16(lay.R, lay.P, lay.rows.ctypes.data_as(_i64p),
                                 lay.row_len.ctypes.data_as(_i64p), _ptrs(pa), _ptrs(sh))
    assert rc == 0
    return list(shards)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening: the bf16 pattern becomes the top half of the fp32 pattern."""
    return (np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def rs_points(lay: Layout, d: np.ndarray, j: np.ndarray,
              fetch: Callable[[int, int, np.ndarray], np.ndarray]) -> np.ndarray:
    """Reduce-scatter outputs ``shard[d[n]][j[n]]`` computed one by one.

    ``fetch(r, p, idx)`` returns the bf16 bits of elements ``idx`` of rank r's gradient of
    parameter p.  The parameter owning shard element j is the last p with o_p <= j; its padded
    row and column follow from j - o_p, and the sum is the same ascending-rank fp32 left fold
    as ``oracle_reduce_scatter``."""
    d = np.asarray(d, np.int64)
    j = np.asarray(j, np.int64)
    out = np.zeros(d.shape, np.float32)
    p_of = np.searchsorted(lay.o, j, side="right") - 1
    for p in np.unique(p_of):
        sel = np.nonzero(p_of == p)[0]
        e = j[sel] - lay.o[p]
        row = d[sel] * lay.m[p] + e // lay.row_len[p]
        valid = row < lay.rows[p]
        idx = row[valid] * lay.row_len[p] + e[valid] % lay.row_len[p]
        acc = bf16_to_f32(fetch(0, int(p), idx))
        for r in range(1, lay.R):
            acc = (acc + bf16_to_f32(fetch(r, int(p), idx))).astype(np.float32)
        vals = np.zeros(sel.size, np.float32)
        vals[valid] = acc
        out[sel] = vals
    return out


def ag_points(lay: Layout, p: int, idx: np.ndarray):
    """Where all-gather output ``param_p[idx]`` comes from: (source rank, element of its shard).

    Element idx of parameter p lies in row idx // L_p; that row belongs to rank row // m_p,
    at padded row row - rank*m_p of its piece, which starts at o_p in the rank's shard."""
    idx = np.asarray(idx, np.int64)
    L, m = int(lay.row_len[p]), int(lay.m[p])
    row = idx // L
    r = row // m
    j = int(lay.o[p]) + (row - r * m) * L + idx % L
    return r, j

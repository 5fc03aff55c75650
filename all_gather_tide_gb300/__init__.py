"""GB300 (sm_103a) layout-aware reduce-scatter and all-gather placement for FSDP2 groups.

A thin ctypes binding of ``libtide.so`` (C ABI in ``include/tide.h``).  Functions carry the C
names; they only marshal arguments (tensors -> device pointers, stream objects -> handles) and
turn negative statuses into :class:`TideError`.  Every step of the path runs in the library's
CUDA kernels or copy-engine calls; there is no Python or CPU fallback, and importing a function
fails loudly if the library has not been built.

"TIDE" is "The Endgame of FSDP Communication: Layout-Aware Collectives on Copy Engines, RDMA, and
NVSwitch" (arXiv 2610.38228): the reduce-scatter is its TIDE-RS (abstract; Fig. 2b), the
placement its TIDE-AG landing (abstract; Fig. 5b), the layout its Table 2.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtide.so")

TIDE_OK = 0
TIDE_EINVAL = -1
TIDE_EALIGN = -2
TIDE_ELAYOUT = -3
TIDE_ECUDA = -4
TIDE_ENOMEM = -5
TIDE_ERANGE = -6
TIDE_FLAG_VEC_STRICT = 0x1
TIDE_FLAG_CE_STRICT = 0x2
TIDE_FLAG_CE_2D = 0x4
TIDE_FLAG_OVERLAP = 0x8
TIDE_FLAG_CE_1D = 0x10
TIDE_RS_AUTO = 0
TIDE_RS_REGISTER = 1
TIDE_RS_BULK = 2
TIDE_RS_TMEM = 3
TIDE_AG_AUTO = 0
TIDE_AG_REGISTER = 1
TIDE_AG_BULK = 2
TIDE_DEBUG_STALL_PRODUCER = 0x1

_lib = None
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
_vpp = ctypes.POINTER(ctypes.c_void_p)

# name -> (restype, argtypes); every symbol declared in include/tide.h
SIGNATURES = {
    "tide_plan_layout": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _i64p, _i64p, _i64p, _i64p, _i64p]),
    "tide_group_create": (ctypes.c_int, [_vpp, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, ctypes.c_uint32]),
    "tide_group_destroy": (ctypes.c_int, [_vp]),
    "tide_group_shard_elems": (ctypes.c_int, [_vp, _i64p]),
    "tide_group_unsharded_elems": (ctypes.c_int, [_vp, _i64p]),
    "tide_group_param_layout": (ctypes.c_int, [_vp, ctypes.c_int32, _i64p, _i64p]),
    "tide_group_valid_rows": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32, _i64p]),
    "tide_group_set_ctas": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32]),
    "tide_group_get_ctas": (ctypes.c_int, [_vp, _i32p, _i32p]),
    "tide_reduce_scatter": (ctypes.c_int, [_vp, _vpp, _vpp, _vp]),
    "tide_reduce_scatter_slots": (ctypes.c_int, [_vp, ctypes.c_int32, _vpp, _vp, _vp]),
    "tide_probe_mixed": (ctypes.c_int, [_vp, ctypes.c_int64, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, _vp, _vp]),
    "tide_stage_slices": (ctypes.c_int, [_vp, ctypes.c_int32, _vpp, _vpp, _vp]),
    "tide_all_gather": (ctypes.c_int, [_vp, _vpp, _vpp, _vp]),
    "tide_all_gather_ce": (ctypes.c_int, [_vp, _vpp, _vpp, _vp]),
    "tide_group_last_ce_copies": (ctypes.c_int, [_vp, _i64p, _i32p]),
    "tide_group_set_rs_variant": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "tide_group_set_ag_variant": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "tide_group_set_ce_lanes": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "tide_group_set_ce_bands": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "tide_group_ag_kernel": (ctypes.c_int, [_vp, _i32p]),
    "tide_group_rs_kernel": (ctypes.c_int, [_vp, _i32p]),
    "tide_group_set_wait_timeout": (ctypes.c_int, [_vp, ctypes.c_uint64]),
    "tide_group_device_status": (ctypes.c_int, [_vp, _i32p]),
    "tide_group_set_debug": (ctypes.c_int, [_vp, ctypes.c_uint32]),
    "tide_reduce_scatter_noalloc": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _vpp, _vpp, _vp]),
    "tide_probe_hold": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64,
                                       _vp, _vp]),
    "tide_probe_bulk_read": (ctypes.c_int, [_vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp]),
    "tide_probe_ingest": (ctypes.c_int, [_vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp]),
    "tide_stage_into_slots": (ctypes.c_int, [_vp, _vpp, _vpp, ctypes.c_int64, _vpp, _vp]),
    "tide_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "tide_last_cuda_error": (ctypes.c_int, []),
    "tide_version": (ctypes.c_int, []),
}


class TideError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().tide_strerror(status).decode()
        if status == TIDE_ECUDA:
            msg += f" (cudaError {lib().tide_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{status}]")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m all_gather_tide_gb300.build` "
                               "(or __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != TIDE_OK:
        raise TideError(status, where)


def _ptr(x) -> int:
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(xs: Sequence) -> ctypes.Array:
    if isinstance(xs, ctypes.Array):  # already marshalled (see pointer_table)
        return xs
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def pointer_table(xs: Sequence) -> ctypes.Array:
    """Marshals tensors (or raw addresses) once into the pointer array the C calls take, for callers
    that pass the same buffers every step: a group with hundreds of parameters otherwise pays about
    a millisecond of Python per call to read R*P data pointers.  The tensors must stay alive and
    unmoved while the table is in use."""
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _i64_array(xs: Sequence[int]):
    return (ctypes.c_int64 * len(xs))(*[int(x) for x in xs])


# ---- C-named functions ------------------------------------------------------------------------


def tide_version() -> int:
    return lib().tide_version()


def tide_strerror(status: int) -> str:
    return lib().tide_strerror(status).decode()


def tide_last_cuda_error() -> int:
    return lib().tide_last_cuda_error()


def tide_plan_layout(R: int, rows: Sequence[int], row_len: Sequence[int]):
    """Host-only planner: returns (m, s, o, S, U) as Python lists / ints."""
    P = len(rows)
    m, s, o = (ctypes.c_int64 * P)(), (ctypes.c_int64 * P)(), (ctypes.c_int64 * P)()
    S, U = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().tide_plan_layout(R, P, _i64_array(rows), _i64_array(row_len), m, s, o,
                                  ctypes.byref(S), ctypes.byref(U)), "tide_plan_layout")
    return list(m), list(s), list(o), S.value, U.value


def tide_group_create(R: int, rows: Sequence[int], row_len: Sequence[int], flags: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(lib().tide_group_create(ctypes.byref(h), R, len(rows), _i64_array(rows), _i64_array(row_len), flags),
           "tide_group_create")
    return h.value


def tide_group_destroy(g: int) -> None:
    _check(lib().tide_group_destroy(g), "tide_group_destroy")


def tide_group_shard_elems(g: int) -> int:
    v = ctypes.c_int64()
    _check(lib().tide_group_shard_elems(g, ctypes.byref(v)), "tide_group_shard_elems")
    return v.value


def tide_group_unsharded_elems(g: int) -> int:
    v = ctypes.c_int64()
    _check(lib().tide_group_unsharded_elems(g, ctypes.byref(v)), "tide_group_unsharded_elems")
    return v.value


def tide_group_param_layout(g: int, p: int) -> Tuple[int, int]:
    m, o = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().tide_group_param_layout(g, p, ctypes.byref(m), ctypes.byref(o)), "tide_group_param_layout")
    return m.value, o.value


def tide_group_valid_rows(g: int, d: int, p: int) -> int:
    v = ctypes.c_int64()
    _check(lib().tide_group_valid_rows(g, d, p, ctypes.byref(v)), "tide_group_valid_rows")
    return v.value


def tide_group_set_ctas(g: int, rs_ctas: int = 0, ag_ctas: int = 0) -> None:
    _check(lib().tide_group_set_ctas(g, rs_ctas, ag_ctas), "tide_group_set_ctas")


def tide_group_get_ctas(g: int) -> Tuple[int, int]:
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().tide_group_get_ctas(g, ctypes.byref(a), ctypes.byref(b)), "tide_group_get_ctas")
    return a.value, b.value


def _flat_grads(grads):
    if isinstance(grads, ctypes.Array):
        return grads
    if len(grads) and isinstance(grads[0], (list, tuple)):
        return [x for row in grads for x in row]
    return list(grads)


def tide_reduce_scatter(g: int, grads, shards: Sequence, stream=None) -> None:
    """``grads``: R lists of P bf16 tensors (or a flat list indexed r*P+p, or raw pointers);
    ``shards``: R fp32 tensors of at least S elements."""
    _check(lib().tide_reduce_scatter(g, _ptr_array(_flat_grads(grads)), _ptr_array(shards), _stream(stream)),
           "tide_reduce_scatter")


def tide_stage_slices(g: int, d: int, grads, slots: Sequence, stream=None) -> None:
    """Copies slice d of every contributor's gradients into ``slots`` (R bf16 tensors of S elements)
    at the shard offsets, one copy-engine copy per (contributor, parameter)."""
    _check(lib().tide_stage_slices(g, d, _ptr_array(_flat_grads(grads)), _ptr_array(slots), _stream(stream)),
           "tide_stage_slices")


def tide_reduce_scatter_slots(g: int, d: int, slots: Sequence, shard, stream=None) -> None:
    """``slots``: R bf16 staging slots of S elements (slot r holds contributor r's slice d of every
    parameter at o_p); ``shard``: d's fp32 shard of S elements."""
    _check(lib().tide_reduce_scatter_slots(g, d, _ptr_array(slots), _ptr(shard), _stream(stream)),
           "tide_reduce_scatter_slots")


def tide_all_gather(g: int, shards: Sequence, params: Sequence, stream=None) -> None:
    _check(lib().tide_all_gather(g, _ptr_array(shards), _ptr_array(params), _stream(stream)), "tide_all_gather")


def tide_all_gather_ce(g: int, shards: Sequence, params: Sequence, stream=None) -> None:
    _check(lib().tide_all_gather_ce(g, _ptr_array(shards), _ptr_array(params), _stream(stream)),
           "tide_all_gather_ce")


def tide_group_set_rs_variant(g: int, variant: int) -> None:
    _check(lib().tide_group_set_rs_variant(g, variant), "tide_group_set_rs_variant")


def tide_group_set_ag_variant(g: int, variant: int) -> None:
    _check(lib().tide_group_set_ag_variant(g, variant), "tide_group_set_ag_variant")


def tide_group_ag_kernel(g: int) -> int:
    v = ctypes.c_int32()
    _check(lib().tide_group_ag_kernel(g, ctypes.byref(v)), "tide_group_ag_kernel")
    return v.value


def tide_group_rs_kernel(g: int) -> int:
    v = ctypes.c_int32()
    _check(lib().tide_group_rs_kernel(g, ctypes.byref(v)), "tide_group_rs_kernel")
    return v.value


def tide_group_set_ce_lanes(g: int, lanes: int) -> None:
    _check(lib().tide_group_set_ce_lanes(g, lanes), "tide_group_set_ce_lanes")


def tide_group_set_ce_bands(g: int, bands: int) -> None:
    _check(lib().tide_group_set_ce_bands(g, bands), "tide_group_set_ce_bands")


def tide_group_set_wait_timeout(g: int, timeout_ns: int) -> None:
    _check(lib().tide_group_set_wait_timeout(g, timeout_ns), "tide_group_set_wait_timeout")


def tide_group_device_status(g: int) -> int:
    v = ctypes.c_int32()
    _check(lib().tide_group_device_status(g, ctypes.byref(v)), "tide_group_device_status")
    return v.value


def tide_group_set_debug(g: int, flags: int) -> None:
    _check(lib().tide_group_set_debug(g, flags), "tide_group_set_debug")


def tide_reduce_scatter_noalloc(R: int, rows: Sequence[int], row_len: Sequence[int], grads, shards: Sequence,
                                stream=None) -> None:
    """Reduce-scatter without any allocation (for callers that cannot allocate device memory):
    the work tables go to the library's fixed device scratch array.  Same data layout as
    ``tide_reduce_scatter``; calls on different streams must not overlap."""
    _check(lib().tide_reduce_scatter_noalloc(R, len(rows), _i64_array(rows), _i64_array(row_len),
                                             _ptr_array(_flat_grads(grads)), _ptr_array(shards), _stream(stream)),
           "tide_reduce_scatter_noalloc")


def tide_stage_into_slots(g: int, grads, slots: Sequence, slot_elems: int, stream=None) -> List[int]:
    """Slot-Reuse staging: copies every rank's gradients into its slot (packed, no padding) and
    returns the R*P staged device addresses (flat, index r*P+p) for ``tide_reduce_scatter``."""
    flat = _flat_grads(grads)
    staged = (ctypes.c_void_p * len(flat))()
    _check(lib().tide_stage_into_slots(g, _ptr_array(flat), _ptr_array(slots), slot_elems, staged, _stream(stream)),
           "tide_stage_into_slots")
    return [int(x) for x in staged]


def tide_group_last_ce_copies(g: int) -> Tuple[int, bool]:
    n, u = ctypes.c_int64(), ctypes.c_int32()
    _check(lib().tide_group_last_ce_copies(g, ctypes.byref(n), ctypes.byref(u)), "tide_group_last_ce_copies")
    return n.value, bool(u.value)


def tide_probe_hold(ctas: int, threads: int, smem_bytes: int, cluster_size: int, hold_ns: int, records=None,
                    stream=None) -> None:
    """Resident probe CTAs (Fig. 4 spin kernels; Table 5 SM-id probe when ``records`` is given:
    a device uint64 tensor of 3*ctas entries receiving SM id, entry and exit ns per CTA)."""
    _check(lib().tide_probe_hold(ctas, threads, smem_bytes, cluster_size, hold_ns,
                                 _ptr(records) if records is not None else None, _stream(stream)), "tide_probe_hold")


def tide_probe_bulk_read(buf, nbytes: int, ctas: int, copy_bytes: int, stages: int, out, stream=None) -> None:
    """Bulk-copy read bandwidth probe; ``out`` is a device uint32/int32 tensor of 2 entries."""
    _check(lib().tide_probe_bulk_read(_ptr(buf), nbytes, ctas, copy_bytes, stages, _ptr(out), _stream(stream)),
           "tide_probe_bulk_read")


def tide_probe_ingest(buf, bulk_bytes: int, ldg_bytes: int, ctas: int, copy_bytes: int, stages: int,
                      consumer_warps: int, ldg_warps: int, out, stream=None) -> None:
    """Per-SM ingest probe (bulk copies read out of shared memory and/or 32-byte register loads);
    ``out`` is a device uint32/int32 tensor of 2 entries."""
    _check(lib().tide_probe_ingest(_ptr(buf), bulk_bytes, ldg_bytes, ctas, copy_bytes, stages, consumer_warps,
                                   ldg_warps, _ptr(out), _stream(stream)), "tide_probe_ingest")


def tide_probe_mixed(buf, bulk_bytes: int, st_buf, st_bytes: int, ctas: int, copy_bytes: int, stages: int,
                     consumer_warps: int, st_warps: int, out, stream=None, burst_rows: int = 0,
                     burst_vecs: int = 0) -> None:
    """Per-SM read/write sharing probe (bulk copies read out of shared memory while other warps
    write 32-byte vectors); ``out`` is a device int64 tensor of 3 entries (checksum, error flags,
    bytes written)."""
    _check(lib().tide_probe_mixed(_ptr(buf), bulk_bytes, _ptr(st_buf) if st_buf is not None else None, st_bytes,
                                  ctas, copy_bytes, stages, consumer_warps, st_warps, burst_rows, burst_vecs,
                                  _ptr(out), _stream(stream)),
           "tide_probe_mixed")


# ---- convenience object -----------------------------------------------------------------------


class Group:
    """Owns one ``tide_group_t``.  ``params`` is a list of ``(rows, row_len)`` pairs."""

    def __init__(self, R: int, params: Sequence[Tuple[int, int]], flags: int = 0):
        self.R = R
        self.rows = [int(r) for r, _ in params]
        self.row_len = [int(l) for _, l in params]
        self.P = len(self.rows)
        self.handle = tide_group_create(R, self.rows, self.row_len, flags)
        self.S = tide_group_shard_elems(self.handle)
        self.U = tide_group_unsharded_elems(self.handle)

    def close(self) -> None:
        if self.handle:
            tide_group_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def param_layout(self, p: int) -> Tuple[int, int]:
        return tide_group_param_layout(self.handle, p)

    def valid_rows(self, d: int, p: int) -> int:
        return tide_group_valid_rows(self.handle, d, p)

    def set_ctas(self, rs_ctas: int = 0, ag_ctas: int = 0) -> None:
        tide_group_set_ctas(self.handle, rs_ctas, ag_ctas)

    def get_ctas(self) -> Tuple[int, int]:
        return tide_group_get_ctas(self.handle)

    def reduce_scatter(self, grads, shards, stream=None) -> None:
        tide_reduce_scatter(self.handle, grads, shards, stream)

    def stage_slices(self, d: int, grads, slots, stream=None) -> None:
        tide_stage_slices(self.handle, d, grads, slots, stream)

    def reduce_scatter_slots(self, d: int, slots, shard, stream=None) -> None:
        tide_reduce_scatter_slots(self.handle, d, slots, shard, stream)

    def all_gather(self, shards, params, stream=None) -> None:
        tide_all_gather(self.handle, shards, params, stream)

    def all_gather_ce(self, shards, params, stream=None) -> None:
        tide_all_gather_ce(self.handle, shards, params, stream)

    def last_ce_copies(self) -> Tuple[int, bool]:
        return tide_group_last_ce_copies(self.handle)

    def stage_into_slots(self, grads, slots, slot_elems: int, stream=None) -> List[int]:
        return tide_stage_into_slots(self.handle, grads, slots, slot_elems, stream)

    def set_rs_variant(self, variant: int) -> None:
        tide_group_set_rs_variant(self.handle, variant)

    def set_ag_variant(self, variant: int) -> None:
        tide_group_set_ag_variant(self.handle, variant)

    def ag_kernel(self) -> int:
        return tide_group_ag_kernel(self.handle)

    def rs_kernel(self) -> int:
        return tide_group_rs_kernel(self.handle)

    def set_ce_lanes(self, lanes: int) -> None:
        tide_group_set_ce_lanes(self.handle, lanes)

    def set_ce_bands(self, bands: int) -> None:
        tide_group_set_ce_bands(self.handle, bands)

    def set_wait_timeout(self, timeout_ns: int) -> None:
        tide_group_set_wait_timeout(self.handle, timeout_ns)

    def device_status(self) -> int:
        return tide_group_device_status(self.handle)

    def set_debug(self, flags: int) -> None:
        tide_group_set_debug(self.handle, flags)

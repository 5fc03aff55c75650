"""Benchmark of the layout-aware reduce-scatter + all-gather placement on one GB300 per process.

A step is one pass of the hot path over one batch of synthetic input: the mixed-precision
reduce-scatter of a whole parameter group (R ranks' bf16 gradients -> R fp32 shards) followed by
the all-gather placement of R packed bf16 shards into per-parameter storage (SM kernel).  The
default workload is the Llama-3.1-70B decoder-layer group at R = 8.  Inputs are resident in HBM
and larger than L2 (17.1 GB of reduce-scatter traffic per step), so no L2 flush is needed.

Printed (rank 0, one JSON line): the effective HBM GB/s of the step (algorithmic bytes / time),
per-leg GB/s and fraction of the measured HBM peak (reduce-scatter, SM placement, copy-engine
placement), the roofline of the dominant kernel (reduce-scatter), the end-to-end figure through
the C ABI with host buffers, how much a single-wave cuBLAS bf16 GEMM (4096 x 4096 x 8192)
running beside the collective on another stream slows down, SM clocks sampled during the timed region, and the CPU
oracle timed on the host on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tide|reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
# The harness runs a collective (up to 8 copy-engine streams) beside a victim on its own stream; with
# the default 8 hardware work queues, streams would share queues and the victim would wait behind
# copies instead of running beside them.  Set before CUDA starts (importing torch does not start it).
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import Group, group, rng  # noqa: E402

METRIC = "RS/AG effective HBM GB/s and % of GB300 peak; concurrent GEMM slowdown %"
FALLBACK_HBM_GBS = 6800.0
DATA = "synthetic (seeded counter-based N(0,1e-3) gradients, N(0,0.02) shards; layer shapes only)"


def workload(args) -> Group:
    g = group(args.workload)
    return g.scaled(args.scale) if args.scale > 1 else g


# ---- layout arithmetic for the byte counts (through the library's host-only planner) ---------


def layout(g: Group):
    import all_gather_tide_gb300 as tide

    m, s, o, S, U = tide.tide_plan_layout(g.R, g.rows, g.row_len)
    return S, U


def workload_config(g: Group, S: int, U: int, replicas: int) -> dict:
    """The workload a step processes, the same dict for the GPU arm and the reference arm."""
    step_bytes = rs_bytes(g, S, U) + ag_bytes(U)
    return {"workload": g.name, "R": g.R, "P": g.P, "U": U, "S": S,
            "step": "reduce-scatter + all-gather placement of the whole group", "step_bytes": step_bytes,
            "l2": f"inputs larger than L2 ({step_bytes / 1e9:.1f} GB of traffic per step), no flush",
            "replicas": replicas}


def rs_bytes(g: Group, S: int, U: int) -> int:
    """Algorithmic reduce-scatter bytes: R*U*2 bf16 read + R*S*4 fp32 written (padding included)."""
    return g.R * U * 2 + g.R * S * 4


def ag_bytes(U: int) -> int:
    """Algorithmic all-gather placement bytes: U*2 read + U*2 written (padding neither)."""
    return 4 * U


# ---- peaks, clocks, profiles -------------------------------------------------------------------


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "all_gather_tide_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, srcs):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != kernel_source_hash(srcs):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.samples = []
        self.proc = None
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu=uuid,{self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        rows = self.samples
        if self.uuid:
            mine = [r for r in rows if self.uuid.replace("GPU-", "") in r[0]]
            if mine:
                rows = mine
        sm = [float(r[1]) for r in rows if len(r) > 7 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 7 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) > 7 for i in range(4) if r[4 + i] == "Active"})
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sm)}


def bind_to_gpu_numa_node(device: int) -> dict:
    """Runs this process on the CPUs next to the GPU, so pinned host buffers are allocated (first
    touch) in the memory attached to them and host<->device copies take the direct link.  Host
    side only; nothing about the GPU changes."""
    info = {"bound": False}
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        q = subprocess.run(["nvidia-smi", "--query-gpu=uuid,pci.bus_id", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=30).stdout
        bus = None
        for line in q.strip().splitlines():
            u, b = [x.strip() for x in line.split(",")]
            if uuid.replace("GPU-", "") in u or len(q.strip().splitlines()) == 1:
                bus = b
        if not bus:
            return info
        dom, rest = bus.split(":", 1)
        sysdir = f"/sys/bus/pci/devices/{dom[-4:].lower()}:{rest.lower()}"
        with open(os.path.join(sysdir, "local_cpulist")) as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        if cpus:
            os.sched_setaffinity(0, cpus)
            info = {"bound": True, "cpus": len(cpus)}
        with open(os.path.join(sysdir, "numa_node")) as f:
            info["numa_node"] = int(f.read().strip())
    except Exception as e:  # no sysfs entry, no nvidia-smi: leave the process as it is
        info["error"] = type(e).__name__
    return info


# ---- multi-process aggregation (one replica per GPU; no data-path collective) ----------------


def max_over_ranks(ms: float, world: int, device) -> float:
    """Slowest rank's elapsed time (ms); the identity at world size 1."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Units all ranks processed / the slowest rank's time, in GB/s."""
    return bytes_per_step * steps * world / (max_ms * 1e-3) / 1e9


# ---- device buffers ----------------------------------------------------------------------------


class Buffers:
    def __init__(self, g: Group, S: int, device):
        self.grads = [[rng.grad_bits(g, r, p, device=device).view(torch.bfloat16) for p in range(g.P)]
                      for r in range(g.R)]
        self.shards = torch.empty(g.R, S, dtype=torch.float32, device=device)
        self.ag_in = torch.stack([rng.shard_bits(g, r, S, device=device) for r in range(g.R)]).view(torch.bfloat16)
        self.params = [torch.empty(g.numel(p), dtype=torch.bfloat16, device=device) for p in range(g.P)]
        self.shard_list = list(self.shards)
        self.ag_list = list(self.ag_in)


# ---- the GPU arm -------------------------------------------------------------------------------


def run_tide(args, rank, world, local_rank):
    import all_gather_tide_gb300 as tide

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    numa = bind_to_gpu_numa_node(local_rank)
    g = workload(args)
    S, U = layout(g)
    G = tide.Group(g.R, list(zip(g.rows, g.row_len)))
    G.set_ctas(args.rs_ctas, args.ag_ctas)
    G.set_rs_variant({"auto": tide.TIDE_RS_AUTO, "register": tide.TIDE_RS_REGISTER,
                      "bulk": tide.TIDE_RS_BULK, "tmem": tide.TIDE_RS_TMEM}[args.rs_variant])
    G.set_ag_variant({"auto": tide.TIDE_AG_AUTO, "register": tide.TIDE_AG_REGISTER,
                      "bulk": tide.TIDE_AG_BULK}[args.ag_variant])
    if args.ce_lanes:
        G.set_ce_lanes(args.ce_lanes)
    rs_ctas, ag_ctas = G.get_ctas()
    buf = Buffers(g, S, dev)
    stream = torch.cuda.Stream(device=dev)
    b_rs, b_ag = rs_bytes(g, S, U), ag_bytes(U)
    peak, peak_kind = hbm_peak()

    def step(ce=False):
        G.reduce_scatter(buf.grads, buf.shard_list, stream)
        (G.all_gather_ce if ce else G.all_gather)(buf.ag_list, buf.params, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    # -- timed region: K steps, events on the launching stream around every kernel -------------
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                ev[k][0].record(stream)
                G.reduce_scatter(buf.grads, buf.shard_list, stream)
                ev[k][1].record(stream)
                G.all_gather(buf.ag_list, buf.params, stream)
                ev[k][2].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(ev[0][0].elapsed_time(ev[-1][2]), world, dev)
    rs_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ag_ms = [e[1].elapsed_time(e[2]) for e in ev]
    ms_per_step = total_ms / args.steps
    step_bytes = b_rs + b_ag
    value = whole_job_gbs(step_bytes, args.steps, world, total_ms)

    rs_avg = statistics.mean(rs_ms)
    ag_avg = statistics.mean(ag_ms)
    legs = {
        "reduce_scatter": {"gbs": b_rs / (rs_avg * 1e-3) / 1e9, "ms": rs_avg, "ms_median": statistics.median(rs_ms),
                           "bytes": b_rs, "ctas": rs_ctas},
        "all_gather_sm": {"gbs": b_ag / (ag_avg * 1e-3) / 1e9, "ms": ag_avg, "ms_median": statistics.median(ag_ms),
                          "bytes": b_ag, "ctas": ag_ctas,
                          "kernel": "all_gather_bulk_kernel" if G.ag_kernel() == tide.TIDE_AG_BULK
                          else "all_gather_kernel"},
    }
    # copy-engine placement and the bulk-copy placement, same buffers (outside the step's timed region)
    legs["all_gather_ce"] = time_ce(G, buf, stream, b_ag, max(3, args.steps))
    G1 = tide.Group(g.R, list(zip(g.rows, g.row_len)), tide.TIDE_FLAG_CE_2D)
    if args.ce_lanes:
        G1.set_ce_lanes(args.ce_lanes)
    G1.set_ce_bands(1)  # the paper's form: one strided copy per parameter
    legs["all_gather_ce_2d"] = time_ce(G1, buf, stream, b_ag, max(3, args.steps))
    # each parameter's strided copy split into bands of ranks, spread over the lanes
    for bands in args.ce_bands_sweep:
        G1.set_ce_bands(bands)
        legs[f"all_gather_ce_2d_bands{bands}"] = time_ce(G1, buf, stream, b_ag, max(3, args.steps))
    G1.set_ce_bands(1)
    for lanes in args.ce_lanes_sweep:
        for name, grp in (("1d", G), ("2d", G1)):
            grp.set_ce_lanes(lanes)
            legs[f"all_gather_ce_{name}_lanes{lanes}"] = time_ce(grp, buf, stream, b_ag, max(3, args.steps))
    if args.ce_lanes_sweep:
        G.set_ce_lanes(args.ce_lanes or 8)
    G1.close()
    legs["all_gather_register"] = time_ag_variant(G, buf, stream, b_ag, max(3, args.steps), args, "register")
    # the summing step always runs the bulk-copy kernel: the caller's count, else one CTA per SM
    slot_ctas = args.rs_ctas or torch.cuda.get_device_properties(dev).multi_processor_count
    legs["reduce_scatter_slots"] = time_rs_slots(G, g, buf, S, stream, max(3, args.steps), slot_ctas,
                                                 "reduce_scatter_bulk_kernel" if G.rs_kernel() == tide.TIDE_RS_BULK
                                                 else "reduce_scatter_tmem_kernel")
    for leg in legs.values():
        leg["frac_of_peak"] = leg["gbs"] / peak

    out = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "io_dtypes": {"grads": "bf16", "rs_shards": "f32", "ag_shards": "bf16", "params": "bf16"},
        "data": DATA,
        "config": workload_config(g, S, U, world),
        "launch": {"rs_ctas": rs_ctas, "ag_ctas": ag_ctas, "step": "tide_reduce_scatter + tide_all_gather (SM kernel)"},
        "legs": legs,
        "gpu_launches": 2 * args.steps,
    }
    # the kernel the library runs for these (16-byte aligned, torch-allocated) gradients
    rs_kernel, rs_srcs = {tide.TIDE_RS_REGISTER: ("reduce_scatter_kernel", ["rs_kernel.cu", "tide_internal.h"]),
                          tide.TIDE_RS_BULK: ("reduce_scatter_bulk_kernel", ["rs_bulk_kernel.cu", "tide_internal.h"]),
                          tide.TIDE_RS_TMEM: ("reduce_scatter_tmem_kernel", ["rs_bulk_kernel.cu", "tide_internal.h"]),
                          }[G.rs_kernel()]
    legs["reduce_scatter"]["kernel"] = rs_kernel
    traffic = recorded_traffic(rs_kernel, g.name, rs_srcs)
    out["roofline"] = {"bound": "hbm", "kernel": rs_kernel, "achieved": legs["reduce_scatter"]["gbs"],
                       "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                       "frac": legs["reduce_scatter"]["gbs"] / peak, "traffic": traffic,
                       "algorithmic_bytes": b_rs}
    out["clocks"] = clocks.summary()

    # end to end first, while nothing but the step has run on the device and the host link
    if not args.no_e2e:
        out["e2e"] = end_to_end(G, g, buf, S, U, dev, args, world)
        out["e2e"]["host_affinity"] = numa
    if args.slot_reuse and rank == 0:
        out["slot_reuse"] = slot_reuse(G, g, buf, S, U, stream)
    if not args.no_stock and rank == 0:
        out["stock_comparator"] = stock_comparator(G, g, buf, S, U, stream, legs)
    if not args.no_interference and rank == 0:
        out["interference"] = interference(G, buf, stream, dev, args)
    if args.probes and rank == 0:
        out["probes"] = probes(G, buf, stream, dev, args)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(g, dev, passes=args.cpu_passes)
    G.close()
    return out


def time_ce(G, buf, stream, b_ag, iters):
    with torch.cuda.stream(stream):
        for _ in range(2):
            G.all_gather_ce(buf.ag_list, buf.params, stream)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(iters)]
        for e in ev:
            e[0].record(stream)
            G.all_gather_ce(buf.ag_list, buf.params, stream)
            e[1].record(stream)
    torch.cuda.synchronize()
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    copies, uniform = G.last_ce_copies()
    avg = statistics.mean(ms)
    return {"gbs": b_ag / (avg * 1e-3) / 1e9, "ms": avg, "ms_median": statistics.median(ms), "bytes": b_ag,
            "copies": copies, "uniform_pitch": uniform, "ctas": 0}


# ---- one-GPU "stock" comparator ----------------------------------------------------------------


def stock_comparator(G, g, buf, S, U, stream, legs):
    """The layout-converting path the paper compares against (Table 1's full-group pack, Table 7's
    copy-out column, Table 8, whose FSDP2 numbers count the _chunk_cat pack), emulated on one GPU with plain
    PyTorch ops (``all_gather_tide_gb300.stock``): every contributor packs its per-parameter bf16
    gradients into a full-group fp32 buffer, the packed buffers are summed per destination (the
    reduce-scatter), and the all-gather output is copied out into padded per-parameter storage.
    Timed with CUDA events; reported against the same algorithmic bytes as the direct path."""
    from all_gather_tide_gb300.stock import StockPath

    sp = StockPath(g.R, g.rows, g.row_len, buf.shards.device)
    out_shards = torch.empty(g.R, S, dtype=torch.float32, device=buf.shards.device)

    def rs():
        sp.reduce_scatter(buf.grads, out_shards)

    def ag():
        sp.copy_out(buf.ag_in)

    def timed(fn, reps=3):
        with torch.cuda.stream(stream):
            fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    rs_ms, ag_ms = timed(rs), timed(ag)
    b_rs, b_ag = rs_bytes(g, S, U), ag_bytes(U)
    # SM time (SMs held x duration), the pages' measure of what a collective takes from compute:
    # the stock ops each fill the GPU; the direct path holds its CTA count (one CTA per SM)
    sms = torch.cuda.get_device_properties(buf.shards.device).multi_processor_count
    rs_ctas0, ag_ctas0 = G.get_ctas()
    G.set_ctas(16, ag_ctas0)
    ms16 = timed(lambda: G.reduce_scatter(buf.grads, buf.shard_list, stream))
    G.set_ctas(rs_ctas0, ag_ctas0)
    direct_ms, direct_ctas = legs["reduce_scatter"]["ms"], legs["reduce_scatter"]["ctas"]
    sm_time = {"stock_sm_ms": rs_ms * sms, "direct_sm_ms": direct_ms * min(direct_ctas, sms),
               "direct_16ctas_ms": ms16, "direct_16ctas_sm_ms": ms16 * 16,
               "ratio_full_width": rs_ms * sms / (direct_ms * min(direct_ctas, sms)),
               "ratio_16ctas": rs_ms * sms / (ms16 * 16)}
    # the direct path's shards (last written by the full-width call above) against the stock sums
    G.reduce_scatter(buf.grads, buf.shard_list, stream)
    torch.cuda.synchronize()
    err = (out_shards - buf.shards).abs().max().item()
    res = {
        "reduce_scatter": {"ms": rs_ms, "gbs_of_direct_bytes": b_rs / (rs_ms * 1e-3) / 1e9,
                           "direct_ms": legs["reduce_scatter"]["ms"], "speedup_direct": rs_ms / legs["reduce_scatter"]["ms"],
                           "extra_buffer_bytes": sp.extra_buffer_bytes,
                           "pack": "torch._chunk_cat" if sp.have_chunk_cat else "chunk+copy",
                           "sm_time": sm_time, "max_abs_diff_vs_direct": err},
        "all_gather_copy_out": {"ms": ag_ms, "gbs_of_direct_bytes": b_ag / (ag_ms * 1e-3) / 1e9,
                                "direct_ms": legs["all_gather_sm"]["ms"], "speedup_direct": ag_ms / legs["all_gather_sm"]["ms"],
                                "op": "torch.split_with_sizes_copy into padded [R, m_p*L_p] storage",
                                # Table 6's SM-ms column: the copy-out fills the GPU, the SM placement
                                # holds its CTAs (at most one per SM), the copy-engine placement no SM
                                "sm_time": {"stock_copy_out_sm_ms": ag_ms * sms,
                                            "direct_sm_sm_ms": legs["all_gather_sm"]["ms"]
                                            * min(legs["all_gather_sm"]["ctas"], sms),
                                            "direct_ce_sm_ms": 0.0}},
    }
    del sp, out_shards
    torch.cuda.empty_cache()
    return res


# ---- Slot-Reuse staging (Fig. 7) ----------------------------------------------------------------


def slot_reuse(G, g, buf, S, U, stream):
    """Slot-Reuse on one GPU: every rank's gradients are copied (copy engines) into an
    all-gather slot no longer in use of R*S bf16 elements, after which the gradient tensors could be released; the
    reduce-scatter then reads the slots.  Reports the staging time, the reduce-scatter from the
    slots, and the gradient bytes that become free once staging is enqueued."""
    slots = torch.empty(g.R, g.R * S, dtype=torch.bfloat16, device=buf.shards.device)
    staged = G.stage_into_slots(buf.grads, list(slots), g.R * S, stream)

    def timed(fn, reps=3):
        with torch.cuda.stream(stream):
            fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    stage_ms = timed(lambda: G.stage_into_slots(buf.grads, list(slots), g.R * S, stream))
    rs_ms = timed(lambda: G.reduce_scatter(staged, buf.shard_list, stream))
    inplace_ms = timed(lambda: G.reduce_scatter(buf.grads, buf.shard_list, stream))
    grad_bytes = g.R * U * 2
    del slots
    torch.cuda.empty_cache()
    return {"stage_ms": stage_ms, "stage_gbs": 2 * grad_bytes / (stage_ms * 1e-3) / 1e9,
            "rs_from_slots_ms": rs_ms, "rs_in_place_ms": inplace_ms,
            "grad_bytes_released_after_staging": grad_bytes, "slot_bytes": g.R * g.R * S * 2}


def time_rs_slots(G, g: Group, buf, S: int, stream, iters: int, ctas: int, kernel: str, d: int = 0) -> dict:
    """The reduce-scatter as destination d would run it on R GPUs: the exchange that fills its R
    staging slots (tide_stage_slices: copy-engine copies, here device to device) and the summing
    step (tide_reduce_scatter_slots) into d's fp32 shard, each timed on its own.  Bytes of the sum:
    the valid slot elements read (2 B each) + S x 4 B written; of the exchange: the same elements
    read and written (2 + 2 B each)."""
    import all_gather_tide_gb300 as tide
    from all_gather_tide_gb300 import exchange

    slots = torch.empty(g.R, S, dtype=torch.bfloat16, device=buf.shards.device)
    out = torch.empty(S, dtype=torch.float32, device=buf.shards.device)
    valid = 0
    for c in exchange.reduce_scatter_pulls(g.R, g.rows, g.row_len, d):
        slots[c.src_rank, c.dst_off:c.dst_off + c.elems].copy_(
            buf.grads[c.src_rank][c.param].view(-1)[c.src_off:c.src_off + c.elems])
        valid += c.elems
    nbytes = valid * 2 + S * 4
    slot_list = list(slots)
    # the exchange, through the library (it rewrites the same elements the copies above wrote)
    grads = tide.pointer_table([t for row in buf.grads for t in row])
    with torch.cuda.stream(stream):
        for _ in range(2):
            G.stage_slices(d, grads, slot_list, stream)
        sev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(iters)]
        for e in sev:
            e[0].record(stream)
            G.stage_slices(d, grads, slot_list, stream)
            e[1].record(stream)
    torch.cuda.synchronize()
    sms = statistics.mean([e[0].elapsed_time(e[1]) for e in sev])
    with torch.cuda.stream(stream):
        for _ in range(2):
            G.reduce_scatter_slots(d, slot_list, out, stream)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(iters)]
        for e in ev:
            e[0].record(stream)
            G.reduce_scatter_slots(d, slot_list, out, stream)
            e[1].record(stream)
    torch.cuda.synchronize()
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    avg = statistics.mean(ms)
    del slots, out, slot_list
    return {"gbs": nbytes / (avg * 1e-3) / 1e9, "ms": avg, "ms_median": statistics.median(ms), "bytes": nbytes,
            "destination": d, "ctas": ctas, "kernel": kernel,
            "what": "tide_reduce_scatter_slots: one destination's R staging slots summed into its fp32 shard",
            "exchange": {"gbs": valid * 4 / (sms * 1e-3) / 1e9, "ms": sms, "bytes": valid * 4,
                         "what": "tide_stage_slices: the R*P copies that fill the slots, copy engines over the "
                                 "group's lanes, device to device on one GPU"}}


def time_ag_variant(G, buf, stream, b_ag, iters, args, variant):
    import all_gather_tide_gb300 as tide

    G.set_ag_variant({"register": tide.TIDE_AG_REGISTER, "bulk": tide.TIDE_AG_BULK}[variant])
    with torch.cuda.stream(stream):
        for _ in range(2):
            G.all_gather(buf.ag_list, buf.params, stream)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(iters)]
        for e in ev:
            e[0].record(stream)
            G.all_gather(buf.ag_list, buf.params, stream)
            e[1].record(stream)
    torch.cuda.synchronize()
    ctas = G.get_ctas()[1]
    G.set_ag_variant({"auto": tide.TIDE_AG_AUTO, "register": tide.TIDE_AG_REGISTER, "bulk": tide.TIDE_AG_BULK}[args.ag_variant])
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    avg = statistics.mean(ms)
    return {"gbs": b_ag / (avg * 1e-3) / 1e9, "ms": avg, "ms_median": statistics.median(ms), "bytes": b_ag,
            "ctas": ctas, "kernel": {"register": "all_gather_kernel", "bulk": "all_gather_bulk_kernel"}[variant]}


# ---- interference harness ----------------------------------------------------------------------


def interference(G, buf, stream, dev, args):
    """Slowdown of a single-wave cuBLAS bf16 GEMM (M=N=4096, K=8192) run on a second stream
    while a collective runs: median(GEMM time inside the collective) / median(alone) - 1."""
    M = N = 4096
    K = 8192
    a = torch.randn(M, K, device=dev, dtype=torch.bfloat16)
    b = torch.randn(K, N, device=dev, dtype=torch.bfloat16)
    c = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
    gs = torch.cuda.Stream(device=dev)

    def gemm():
        torch.matmul(a, b, out=c)

    with torch.cuda.stream(gs):
        for _ in range(10):
            gemm()
        alone_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(50)]
        for e in alone_ev:
            e[0].record(gs)
            gemm()
            e[1].record(gs)
    torch.cuda.synchronize()
    alone = [e[0].elapsed_time(e[1]) for e in alone_ev]
    t_alone = statistics.median(alone)

    def concurrent(launch, label, reps=4):
        """GEMMs back to back on the second stream from the collective's start; a GEMM counts if it
        starts while the collective runs, and its time includes any wait for free SMs."""
        inside = []
        coll_ms = []
        done_inside, window = [0], [0.0]
        for _ in range(reps):
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            with torch.cuda.stream(stream):
                launch()
            s1.record(stream)
            gs.wait_event(s0)
            n = 64
            ge = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
            with torch.cuda.stream(gs):
                for e in ge:
                    e[0].record(gs)
                    gemm()
                    e[1].record(gs)
            torch.cuda.synchronize()
            end = s0.elapsed_time(s1)
            coll_ms.append(end)
            for e in ge:
                if 0 <= s0.elapsed_time(e[0]) < end:
                    inside.append(e[0].elapsed_time(e[1]))
                if s0.elapsed_time(e[1]) <= end:
                    done_inside[0] += 1
            # the rate is taken over the part of the window in which GEMMs were queued
            window[0] += min(end, s0.elapsed_time(ge[-1][1]))
        res = {"collective_ms": statistics.median(coll_ms), "gemms_started_inside": len(inside),
               # GEMM work finished inside the collective's window, as a fraction of what the GEMM
               # alone would finish in that time (1.0 = unaffected; also captures GEMMs kept waiting)
               "victim_rate": done_inside[0] * t_alone / window[0] if window[0] else None}
        if inside:
            res["gemm_ms"] = statistics.median(inside)
            res["slowdown_pct"] = 100.0 * (statistics.median(inside) / t_alone - 1.0)
        else:
            res["slowdown_pct"] = None
        return res

    out = {"gemm": {"M": M, "N": N, "K": K, "dtype": "bf16", "alone_ms": t_alone,
                    "tflops": 2 * M * N * K / (t_alone * 1e-3) / 1e12, "library": "cuBLAS via torch.matmul"}}
    if args.sweep:
        out["cta_sweep"] = cta_sweep(G, buf, stream, args, concurrent)
    rs_default, ag_default = G.get_ctas()
    b_rs, b_ag = rs_bytes_of(G), 4 * G.U
    peak, peak_kind = hbm_peak()

    def alone_ms(launch, reps=2):
        with torch.cuda.stream(stream):
            launch()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                launch()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    out["reduce_scatter"] = dict(ctas=rs_default, **concurrent(lambda: G.reduce_scatter(buf.grads, buf.shard_list, stream), "rs"))
    # the reduce-scatter at capped CTA counts: bandwidth alone and beside the GEMM, and the GEMM's
    # slowdown; the operating point is the largest count that keeps the slowdown <= 10 %
    rs_rows = []
    for n_ctas in args.interference_ctas:
        G.set_ctas(n_ctas, 0)
        launch = lambda: G.reduce_scatter(buf.grads, buf.shard_list, stream)
        ms = alone_ms(launch)
        conc = concurrent(launch, "rs")
        row = dict(ctas=n_ctas, gbs_alone=b_rs / (ms * 1e-3) / 1e9,
                   gbs_beside_gemm=b_rs / (conc["collective_ms"] * 1e-3) / 1e9, **conc)
        out[f"reduce_scatter_ctas{n_ctas}"] = row
        rs_rows.append(row)
    G.set_ctas(args.rs_ctas, args.ag_ctas)
    ok = [r for r in rs_rows if r["slowdown_pct"] is not None and r["slowdown_pct"] <= 10.0]
    if ok:
        best = max(ok, key=lambda r: r["gbs_beside_gemm"])
        out["operating_point"] = {
            "ctas": best["ctas"], "gemm_slowdown_pct": best["slowdown_pct"], "victim_rate": best["victim_rate"],
            "rs_gbs_beside_gemm": best["gbs_beside_gemm"], "frac_beside_gemm": best["gbs_beside_gemm"] / peak,
            "rs_gbs_alone": best["gbs_alone"], "frac_alone": best["gbs_alone"] / peak, "peak": peak,
            "peak_kind": peak_kind, "target_frac": 0.75, "target_slowdown_pct": 10.0,
            "joint_target_met": bool(best["gbs_beside_gemm"] / peak >= 0.75),
            "rule": "largest reduce-scatter bandwidth beside the GEMM among the CTA counts with <= 10 % slowdown"}
    # what 16 SMs could move at best: the measured per-SM ingest ceiling x 16, scaled from bytes
    # read to the reduce-scatter's algorithmic bytes (reads R*U*2 of the R*U*2 + R*S*4)
    ing = sm_ingest(dev, stream, ctas=16)
    read_bytes = 2 * G.R * G.U
    bound = 16 * ing["ceiling_gbs_per_sm"] * b_rs / read_bytes
    out["sm_ingest_16_ctas"] = ing
    mixed = sm_mixed(dev, stream, ctas=16)
    out["sm_mixed_16_ctas"] = mixed
    if "operating_point" in out:
        # the tighter bound: reads and writes share an SM's traffic, and the reduce-scatter writes
        # R*S*4 bytes for every R*U*2 it reads
        per_sm, rd = mixed_bound(mixed["rows"], (b_rs - read_bytes) / read_bytes)
        if per_sm is not None:
            out["operating_point"]["bound_16_sms_mixed_gbs"] = 16 * per_sm
            out["operating_point"]["bound_16_sms_mixed_frac"] = 16 * per_sm / peak
            out["operating_point"]["rs_alone_over_mixed_bound"] = out["operating_point"]["rs_gbs_alone"] / (16 * per_sm)
            out["operating_point"]["bound_mixed_rule"] = (
                "16 x the bytes one SM moves at the reduce-scatter's ratio of bytes written to bytes read, "
                "interpolated between tide_probe_mixed's measured (read, write) points")
        out["operating_point"]["bound_16_sms_gbs"] = bound
        out["operating_point"]["bound_16_sms_frac"] = bound / peak
        out["operating_point"]["bound_rule"] = ("16 x the most bytes per second any ingest-probe mode brought into "
                                                "one SM x (algorithmic bytes / bytes read): the reduce-scatter must "
                                                "bring its inputs into the SMs that run it")
    # the placement is short; run it several times back to back so GEMMs fit inside
    out["all_gather_sm"] = dict(ctas=ag_default, **concurrent(
        lambda: [G.all_gather(buf.ag_list, buf.params, stream) for _ in range(8)], "ag"))
    out["all_gather_ce"] = dict(ctas=0, **concurrent(
        lambda: [G.all_gather_ce(buf.ag_list, buf.params, stream) for _ in range(8)], "ce"))
    # the same copies over a single stream: fewer in flight, much less HBM/L2 contention
    G.set_ce_lanes(1)
    out["all_gather_ce_lanes1"] = dict(ctas=0, ce_lanes=1, **concurrent(
        lambda: [G.all_gather_ce(buf.ag_list, buf.params, stream) for _ in range(8)], "ce"))
    G.set_ce_lanes(args.ce_lanes or 8)
    # plain calls on a group created with TIDE_FLAG_OVERLAP (interference-first defaults)
    import all_gather_tide_gb300 as tide

    Gov = tide.Group(G.R, list(zip(G.rows, G.row_len)), tide.TIDE_FLAG_OVERLAP)
    ov_rs, ov_ag = Gov.get_ctas()
    legs = (("reduce_scatter", lambda: Gov.reduce_scatter(buf.grads, buf.shard_list, stream), b_rs, ov_rs),
            ("all_gather_sm", lambda: [Gov.all_gather(buf.ag_list, buf.params, stream) for _ in range(8)], 8 * b_ag,
             ov_ag),
            ("all_gather_ce", lambda: [Gov.all_gather_ce(buf.ag_list, buf.params, stream) for _ in range(8)],
             8 * b_ag, 0))
    ov = {}
    for name, launch, nbytes, ctas in legs:
        ms = alone_ms(launch)
        conc = concurrent(launch, name)
        ov[name] = dict(ctas=ctas, gbs_alone=nbytes / (ms * 1e-3) / 1e9, frac_alone=nbytes / (ms * 1e-3) / 1e9 / peak,
                        gbs_beside_gemm=nbytes / (conc["collective_ms"] * 1e-3) / 1e9, **conc)
    ov["all_gather_sm"]["kernel"] = "all_gather_bulk_kernel" if Gov.ag_kernel() == tide.TIDE_AG_BULK else "all_gather_kernel"
    ov["all_gather_ce"]["copies"], ov["all_gather_ce"]["uniform_pitch"] = Gov.last_ce_copies()
    # one layer's reduce-scatter and another's all-gather at once, as FSDP overlaps them: the
    # reduce-scatter on its 16 CTAs and copy-engine placements on a second stream until it ends
    s_b = torch.cuda.Stream(device=dev)
    ce_ms = alone_ms(lambda: Gov.all_gather_ce(buf.ag_list, buf.params, stream))
    n_ce = max(1, int(round(ov["reduce_scatter"]["collective_ms"] / max(ce_ms, 1e-3))))

    def both():
        start = torch.cuda.Event()
        start.record(stream)
        s_b.wait_event(start)
        Gov.reduce_scatter(buf.grads, buf.shard_list, stream)
        with torch.cuda.stream(s_b):
            for _ in range(n_ce):
                Gov.all_gather_ce(buf.ag_list, buf.params, s_b)
        end = torch.cuda.Event()
        end.record(s_b)
        stream.wait_event(end)

    ms = alone_ms(both)
    conc = concurrent(both, "rs+ce")
    nbytes = b_rs + n_ce * b_ag
    ov["reduce_scatter_with_ce_placement"] = dict(
        placements=n_ce, gbs_alone=nbytes / (ms * 1e-3) / 1e9,
        gbs_beside_gemm=nbytes / (conc["collective_ms"] * 1e-3) / 1e9, **conc)
    ov["flag"] = "TIDE_FLAG_OVERLAP"
    out["overlap_mode"] = ov
    Gov.close()
    if args.overlap_ce_forms:
        # the copy-engine placement over overlap mode's one lane in each form, whatever the rule picks
        forms = {}
        for form, extra in (("1d", tide.TIDE_FLAG_CE_1D), ("2d", tide.TIDE_FLAG_CE_2D)):
            Gf = tide.Group(G.R, list(zip(G.rows, G.row_len)), tide.TIDE_FLAG_OVERLAP | extra)
            launch = lambda: [Gf.all_gather_ce(buf.ag_list, buf.params, stream) for _ in range(8)]
            ms = alone_ms(launch)
            conc = concurrent(launch, "ce")
            forms[form] = dict(gbs_alone=8 * b_ag / (ms * 1e-3) / 1e9,
                               gbs_beside_gemm=8 * b_ag / (conc["collective_ms"] * 1e-3) / 1e9, **conc)
            forms[form]["copies"], forms[form]["uniform_pitch"] = Gf.last_ce_copies()
            Gf.close()
        out["overlap_ce_forms"] = forms
    return out


def sm_ingest(dev, stream, full=False, ctas=16):
    """Bytes per second one SM can bring in (tide_probe_ingest, `ctas` CTAs, one per SM, over a
    4 GiB buffer): bulk copies alone, bulk copies read out of shared memory, 32-byte register loads,
    and both at once.  The largest is the ceiling of any kernel that reads its inputs through that
    many SMs."""
    import all_gather_tide_gb300 as tide

    nb = 4 << 30
    buf = torch.empty(nb // 4, dtype=torch.int32, device=dev)
    buf.fill_(0x3C00_3C00)
    out = torch.zeros(2, dtype=torch.int32, device=dev)
    cases = [("bulk copies only", 73728, 3, 0, 0, 1.0), ("bulk copies read out", 46080, 5, 15, 0, 1.0),
             ("bulk copies read out", 73728, 3, 15, 0, 1.0), ("register loads only", 32768, 1, 1, 14, 0.0),
             ("both", 65536, 3, 8, 7, 0.6), ("both", 65536, 3, 8, 7, 0.7)]
    if full:
        cases += [("bulk copies only", 46080, 5, 0, 0, 1.0), ("bulk copies read out", 57344, 4, 14, 0, 1.0),
                  ("bulk copies read out", 65536, 3, 15, 0, 1.0), ("register loads only", 32768, 1, 1, 8, 0.0),
                  ("both", 65536, 3, 11, 4, 0.8)]

    def launch(copy, stages, cons, ldgw, f):
        bulk = int(nb * f) // copy * copy
        ldg = (nb - (bulk + 255) // 256 * 256) // 32 * 32 if ldgw else 0
        tide.tide_probe_ingest(buf, bulk, ldg, ctas, copy, stages, cons, ldgw, out, stream)
        return bulk + ldg

    with torch.cuda.stream(stream):
        for _ in range(30):  # bring the clocks up
            launch(73728, 3, 15, 0, 1.0)
    torch.cuda.synchronize()
    rows = []
    for name, copy, stages, cons, ldgw, f in cases:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            launch(copy, stages, cons, ldgw, f)
            ev[0].record(stream)
            n = sum(launch(copy, stages, cons, ldgw, f) for _ in range(3))
            ev[1].record(stream)
        torch.cuda.synchronize()
        gbs = n / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9
        rows.append({"mode": name, "copy_bytes": copy, "stages": stages, "consumer_warps": cons,
                     "ldg_warps": ldgw, "bulk_fraction": f, "gbs": gbs, "gbs_per_sm": gbs / ctas})
    flags = int(out[1].item())  # nonzero: a bounded probe wait expired (the rates are then suspect)
    del buf
    torch.cuda.empty_cache()
    best = max(rows, key=lambda r: r["gbs_per_sm"])
    return {"ctas": ctas, "rows": rows, "ceiling_gbs_per_sm": best["gbs_per_sm"], "ceiling_mode": best["mode"],
            "probe_error_flags": flags}


def sm_mixed(dev, stream, ctas=16):
    """How reads and writes share one SM (tide_probe_mixed, `ctas` CTAs, one per SM): 32-byte
    stores alone, bulk copies read out of shared memory alone, and both at once with 1 to 7 of the
    CTA's 16 warps writing.  A reduce-scatter over R = 8 ranks writes 4 bytes per 16 read."""
    import all_gather_tide_gb300 as tide

    nb, ns = 2 << 30, 1 << 30
    buf = torch.empty(nb // 4, dtype=torch.int32, device=dev)
    buf.fill_(0x3C00_3C00)
    st = torch.empty(ns, dtype=torch.uint8, device=dev)
    out = torch.zeros(3, dtype=torch.int64, device=dev)
    # (mode, copy bytes, stages, reading warps, writing warps, reads?, burst rows, burst vectors)
    cases = [("writes only", 73728, 3, 1, 14, False), ("writes only", 73728, 3, 1, 4, False),
             ("reads only", 73728, 3, 15, 0, True), ("reads and writes", 73728, 3, 14, 1, True),
             ("reads and writes", 73728, 3, 13, 2, True), ("reads and writes", 73728, 3, 12, 3, True),
             ("reads and writes", 73728, 3, 11, 4, True),
             ("reads and writes", 73728, 3, 8, 7, True), ("reads only", 46080, 5, 15, 0, True),
             ("reads and writes", 46080, 5, 14, 1, True),
             # the reading threads themselves store 6 (10) 32-byte vectors after every 8 landed copies:
             # the reduce-scatter's 1:4 ratio and its store pattern at 45 KB (72 KB) copies
             ("reads with burst writes", 46080, 5, 15, 0, True, 8, 6),
             ("reads with burst writes", 73728, 3, 15, 0, True, 8, 10)]
    cases = [c if len(c) == 8 else c + (0, 0) for c in cases]

    def launch(copy, stages, cons, stw, reads, brows=0, bvecs=0):
        bulk = nb // copy * copy if reads else 0
        tide.tide_probe_mixed(buf, bulk, st, ns, ctas, copy, stages, cons, stw, out, stream, brows, bvecs)
        return bulk

    with torch.cuda.stream(stream):
        for _ in range(10):  # bring the clocks up
            launch(73728, 3, 15, 0, True)
    torch.cuda.synchronize()
    rows = []
    for name, copy, stages, cons, stw, reads, brows, bvecs in cases:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            launch(copy, stages, cons, stw, reads, brows, bvecs)
            out[2].zero_()
            ev[0].record(stream)
            n = sum(launch(copy, stages, cons, stw, reads, brows, bvecs) for _ in range(3))
            ev[1].record(stream)
        torch.cuda.synchronize()
        s = ev[0].elapsed_time(ev[1]) * 1e-3
        w = int(out[2].item())
        rows.append({"mode": name, "copy_bytes": copy, "stages": stages, "consumer_warps": cons, "st_warps": stw,
                     "burst_rows": brows, "burst_vecs": bvecs,
                     "read_gbs_per_sm": n / s / 1e9 / ctas, "write_gbs_per_sm": w / s / 1e9 / ctas})
    flags = int(out[1].item())  # nonzero: a bounded probe wait expired (the rates are then suspect)
    del buf, st
    torch.cuda.empty_cache()
    return {"ctas": ctas, "rows": rows, "probe_error_flags": flags}


def mixed_bound(rows, write_per_read: float):
    """Bytes per second (read + written) one SM can move at a given ratio of bytes written to bytes
    read, interpolated between the probe's measured points of the 72 KB x 3 geometry (reads alone,
    then 1, 2, 3, 4 and 7 writer warps), linear in the ratio; None outside the measured range."""
    pts = sorted((r["write_gbs_per_sm"] / r["read_gbs_per_sm"], r["read_gbs_per_sm"]) for r in rows
                 if r["copy_bytes"] == 73728 and r["read_gbs_per_sm"] > 0 and not r.get("burst_rows"))
    for (x0, r0), (x1, r1) in zip(pts, pts[1:]):
        if x0 <= write_per_read <= x1:
            rd = r0 + (r1 - r0) * (write_per_read - x0) / (x1 - x0) if x1 > x0 else min(r0, r1)
            return rd * (1.0 + write_per_read), rd
    return None, None


def cta_sweep(G, buf, stream, args, concurrent):
    """Collective bandwidth alone and concurrent-GEMM slowdown per CTA count (the Pareto curve
    between collective speed and interference; Fig. 4 and Table 4 of the paper)."""
    g_rs = rs_bytes_of(G)
    g_ag = 4 * G.U
    import all_gather_tide_gb300 as tide

    rows = []
    cases = [("reduce_scatter", v, n) for v in (tide.TIDE_RS_REGISTER, tide.TIDE_RS_BULK, tide.TIDE_RS_TMEM)
             for n in args.sweep_rs]
    cases += [("all_gather_sm", v, n) for v in (tide.TIDE_AG_REGISTER, tide.TIDE_AG_BULK) for n in args.sweep_ag]
    for kind, variant, n in cases:
        if kind == "reduce_scatter":
            G.set_ctas(n, 0)
            G.set_rs_variant(variant)
            launch = lambda: G.reduce_scatter(buf.grads, buf.shard_list, stream)
            nbytes, reps = g_rs, 1
        else:
            G.set_ctas(0, n)
            G.set_ag_variant(variant)
            launch = lambda: [G.all_gather(buf.ag_list, buf.params, stream) for _ in range(8)]
            nbytes, reps = g_ag * 8, 8
        with torch.cuda.stream(stream):
            launch()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        c = concurrent(launch, kind, reps=2)
        rows.append({"kind": kind, "variant": {0: "auto", 1: "register", 2: "bulk", 3: "tmem"}[variant], "ctas": n,
                     "alone_ms": ms / reps, "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "gemm_slowdown_pct": c["slowdown_pct"], "gemms": c["gemms_started_inside"]})
    G.set_ctas(args.rs_ctas, args.ag_ctas)
    G.set_rs_variant(tide.TIDE_RS_AUTO)
    G.set_ag_variant(tide.TIDE_AG_AUTO)
    # copy-engine placement: no SM is taken, so the only knob is how many copies run at once
    # (the streams they are spread over); HBM and L2 contention is what slows the GEMM
    G2 = tide.Group(G.R, list(zip(G.rows, G.row_len)), tide.TIDE_FLAG_CE_2D)
    G2.set_ce_bands(1)  # the paper's form: one strided copy per parameter
    for form, grp in (("1d", G), ("2d", G2)):
        for lanes in (1, 2, 4, 8):
            grp.set_ce_lanes(lanes)
            launch = lambda: [grp.all_gather_ce(buf.ag_list, buf.params, stream) for _ in range(8)]
            with torch.cuda.stream(stream):
                launch()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            c = concurrent(launch, "ce", reps=2)
            rows.append({"kind": "all_gather_ce", "variant": form, "ce_lanes": lanes, "ctas": 0,
                         "alone_ms": ms / 8, "gbs": g_ag * 8 / (ms * 1e-3) / 1e9,
                         "gemm_slowdown_pct": c["slowdown_pct"], "victim_rate": c["victim_rate"],
                         "gemms": c["gemms_started_inside"]})
    G.set_ce_lanes(args.ce_lanes or 8)
    G2.close()
    return rows


def rs_bytes_of(G) -> int:
    return G.R * G.U * 2 + G.R * G.S * 4


# ---- interference probes: spin-CTA curve, SM-id probe, victims of Table 4 ---------------------


def _window_times(launch_a, b_stream, victim, n_victims, a_stream):
    """Launch `launch_a` on a_stream and n_victims victims back to back on b_stream from the same
    start; returns (a's elapsed ms, victim ms list for victims that started inside a's window)."""
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(a_stream)
    with torch.cuda.stream(a_stream):
        launch_a()
    s1.record(a_stream)
    b_stream.wait_event(s0)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_victims)]
    with torch.cuda.stream(b_stream):
        for e in ev:
            e[0].record(b_stream)
            victim()
            e[1].record(b_stream)
    torch.cuda.synchronize()
    end = s0.elapsed_time(s1)
    inside = [e[0].elapsed_time(e[1]) for e in ev if 0 <= s0.elapsed_time(e[0]) < end]
    return end, inside


def probes(G, buf, stream, dev, args):
    """Fig. 4 (GEMM slowdown vs resident spin CTAs), Table 5 (SM-id probe: probe CTAs displaced past
    the first wave and SMs held by the collective) and Table 4 (slowdown of a 1-wave GEMM, a 28-wave
    GEMM and an elementwise kernel beside the reduce-scatter), on one GB300."""
    import all_gather_tide_gb300 as tide

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    vs = torch.cuda.Stream(device=dev)
    a1 = torch.randn(4096, 8192, device=dev, dtype=torch.bfloat16)
    b1 = torch.randn(8192, 4096, device=dev, dtype=torch.bfloat16)
    c1 = torch.empty(4096, 4096, device=dev, dtype=torch.bfloat16)
    a2 = torch.randn(16384, 8192, device=dev, dtype=torch.bfloat16)
    b2 = torch.randn(8192, 8192, device=dev, dtype=torch.bfloat16)
    c2 = torch.empty(16384, 8192, device=dev, dtype=torch.bfloat16)
    x = torch.randn(1 << 28, device=dev)
    y = torch.randn(1 << 28, device=dev)
    z = torch.empty(1 << 28, device=dev)
    victims = {
        "gemm_1wave_4096x4096x8192": lambda: torch.matmul(a1, b1, out=c1),
        "gemm_28wave_16384x8192x8192": lambda: torch.matmul(a2, b2, out=c2),
        "elementwise_add_1GiB": lambda: torch.add(x, y, out=z),
    }

    def alone(fn, n=20):
        with torch.cuda.stream(vs):
            for _ in range(3):
                fn()
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
            for e in ev:
                e[0].record(vs)
                fn()
                e[1].record(vs)
        torch.cuda.synchronize()
        return statistics.median(e[0].elapsed_time(e[1]) for e in ev)

    t_alone = {k: alone(f) for k, f in victims.items()}
    out = {"sms": sms, "victims_alone_ms": t_alone}

    # Fig. 4: resident CTAs that fill an SM each (the whole register file and 213 KB of shared
    # memory, like a GEMM CTA)
    curve = []
    g1 = victims["gemm_1wave_4096x4096x8192"]
    for n in args.spin_ctas:
        hold = lambda: tide.tide_probe_hold(n, 1024, 213 * 1024, 1, 20_000_000, None, stream)
        _, inside = _window_times(hold, vs, g1, 64, stream)
        curve.append({"resident_ctas": n, "gemms": len(inside),
                      "slowdown_pct": 100 * (statistics.median(inside) / t_alone["gemm_1wave_4096x4096x8192"] - 1)
                      if inside else None})
    out["spin_curve"] = curve
    # the same resident CTAs launched as clusters: does packing them into whole cluster slots leave
    # the GEMM more room?
    clustered = []
    for cl in (2, 4, 8):
        for n in (16, 20, 24, 32):
            if n % cl:
                continue  # whole clusters only
            hold = lambda: tide.tide_probe_hold(n, 1024, 213 * 1024, cl, 20_000_000, None, stream)
            _, inside = _window_times(hold, vs, g1, 64, stream)
            clustered.append({"cluster": cl, "resident_ctas": n, "gemms": len(inside),
                              "slowdown_pct": 100 * (statistics.median(inside) / t_alone["gemm_1wave_4096x4096x8192"] - 1)
                              if inside else None})
    out["spin_curve_clustered"] = clustered

    # Table 4 / Table 5 for several reduce-scatter configurations, and for the copy-engine
    # placement (8 placements back to back, so the victims and probes overlap it)
    configs = [("reduce_scatter", "tmem", 0), ("reduce_scatter", "tmem", 16), ("reduce_scatter", "tmem", 4),
               ("reduce_scatter", "bulk", 16), ("reduce_scatter", "register", 16), ("all_gather_ce", "1d", 1),
               ("all_gather_ce", "1d", 8),
               ("all_gather_ce", "2d", 1)]
    G2 = tide.Group(G.R, list(zip(G.rows, G.row_len)), tide.TIDE_FLAG_CE_2D)
    G2.set_ce_bands(1)  # the paper's form: one strided copy per parameter
    rows = []
    recs = torch.zeros(3 * sms, dtype=torch.int64, device=dev)
    for coll, variant, n_ in configs:
        if coll == "reduce_scatter":
            G.set_ctas(n_, 0)
            G.set_rs_variant({"bulk": tide.TIDE_RS_BULK, "tmem": tide.TIDE_RS_TMEM,
                              "register": tide.TIDE_RS_REGISTER}[variant])
            rs = lambda: G.reduce_scatter(buf.grads, buf.shard_list, stream)
            row = {"collective": coll, "variant": variant, "ctas": n_ or G.get_ctas()[0]}
        else:
            grp = G if variant == "1d" else G2
            grp.set_ce_lanes(n_)
            rs = lambda: [grp.all_gather_ce(buf.ag_list, buf.params, stream) for _ in range(8)]
            row = {"collective": coll, "variant": variant, "ctas": 0, "ce_lanes": n_}
        for name, fn in victims.items():
            ms, inside = _window_times(rs, vs, fn, 48, stream)
            row["coll_ms"] = ms
            if coll == "reduce_scatter":
                row["rs_ms"] = ms
            row[name] = 100 * (statistics.median(inside) / t_alone[name] - 1) if inside else None
        # SM-id probes: 32 four-CTA clusters (the GEMM's shape) and one CTA per SM, 50 us each,
        # launched repeatedly while the reduce-scatter runs
        disp, res = [], []
        for shape in ("clusters", "per_sm"):
            n, cl = (128, 4) if shape == "clusters" else (sms, 1)
            launches = []

            def probe_many():
                for _ in range(6):
                    tide.tide_probe_hold(n, 1024, 213 * 1024, cl, 50_000, recs, vs)
                    launches.append(recs[:3 * n].clone().view(n, 3))

            torch.cuda.synchronize()
            s0 = torch.cuda.Event()
            s0.record(stream)
            with torch.cuda.stream(stream):
                rs()
            vs.wait_event(s0)
            with torch.cuda.stream(vs):
                probe_many()
            torch.cuda.synchronize()
            for rec in launches:
                entry = rec[:, 1].double()
                late = int((entry > entry.min() + 25_000).sum())  # started after the first wave
                (disp if shape == "clusters" else res).append(late)
        row["probe_displaced_ctas_mode"] = statistics.mode(disp)
        row["probe_windows_hit_pct"] = 100.0 * sum(d > 0 for d in disp) / len(disp)
        row["probe_resident_ctas_mean"] = statistics.mean(res)
        rows.append(row)
    G.set_ctas(args.rs_ctas, args.ag_ctas)
    G.set_rs_variant(tide.TIDE_RS_AUTO)
    G.set_ce_lanes(args.ce_lanes or 8)
    G2.close()
    out["table4_table5"] = rows
    out["sm_ingest"] = {n: sm_ingest(dev, stream, full=True, ctas=n) for n in (16, sms)}
    del a2, b2, c2, x, y, z
    torch.cuda.empty_cache()
    return out


# ---- end to end with host buffers --------------------------------------------------------------


def end_to_end(G, g, buf, S, U, dev, args, world):
    """Same step through the public API with host buffers: every step copies all its inputs in
    from pinned host memory and all its outputs back, inside the timed region.  Input copies are
    spread over several streams (several copy engines), and step k+1's input copies overlap step
    k's output copies (opposite directions of the host link).  The steps alternate between two sets
    of device buffers, so step k+1's input copies also overlap step k's kernels; events keep every
    buffer's reuse ordered after its last reader.  The same loop over one device set is reported
    beside it."""
    h_grads = [[t.to("cpu").pin_memory() for t in row] for row in buf.grads]
    h_ag = buf.ag_in.to("cpu").pin_memory()
    h_shards = torch.empty(g.R, S, dtype=torch.float32).pin_memory()
    h_params = [torch.empty(g.numel(p), dtype=torch.bfloat16).pin_memory() for p in range(g.P)]
    h2d = sum(t.numel() * 2 for row in h_grads for t in row) + h_ag.numel() * 2
    d2h = h_shards.numel() * 4 + sum(t.numel() * 2 for t in h_params)
    sets = [buf, Buffers(g, S, dev)]  # the second set's contents are overwritten by the copies
    n_in = 4
    s_in = [torch.cuda.Stream(device=dev) for _ in range(n_in)]
    s_c = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def plan_lanes(b):
        pairs = [(b.grads[r][p], h_grads[r][p]) for r in range(g.R) for p in range(g.P)] + [(b.ag_in, h_ag)]
        pairs.sort(key=lambda x: -x[0].numel())
        lanes, load = [[] for _ in range(n_in)], [0] * n_in
        for d_t, h_t in pairs:  # balance the bytes over the input streams
            k = load.index(min(load))
            lanes[k].append((d_t, h_t))
            load[k] += d_t.numel()
        return lanes

    lanes = [plan_lanes(b) for b in sets]
    outs = [[(h_shards, b.shards)] + [(h_params[p], b.params[p]) for p in range(g.P)] for b in sets]
    state = {"k": 0, "computed": [None, None], "copied_out": [None, None]}

    def step(nsets):
        k = state["k"] % nsets
        state["k"] += 1
        b = sets[k]
        for i in range(n_in):
            if state["computed"][k] is not None:
                s_in[i].wait_event(state["computed"][k])  # the set's last kernels have read its inputs
            with torch.cuda.stream(s_in[i]):
                for d_t, h_t in lanes[k][i]:
                    d_t.copy_(h_t, non_blocking=True)
        for i in range(n_in):
            s_c.wait_stream(s_in[i])
        if state["copied_out"][k] is not None:
            s_c.wait_event(state["copied_out"][k])  # the set's last outputs have been copied out
        G.reduce_scatter(b.grads, b.shard_list, s_c)
        G.all_gather(b.ag_list, b.params, s_c)
        computed = torch.cuda.Event()
        computed.record(s_c)
        s_out.wait_event(computed)
        with torch.cuda.stream(s_out):
            for h_t, d_t in outs[k]:
                h_t.copy_(d_t, non_blocking=True)
        copied_out = torch.cuda.Event()
        copied_out.record(s_out)
        state["computed"][k], state["copied_out"][k] = computed, copied_out

    def one_direction(direction):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s_c)
        for i in range(n_in):
            s_in[i].wait_event(e0)
            with torch.cuda.stream(s_in[i]):
                for d_t, h_t in lanes[0][i]:
                    if direction == "h2d":
                        d_t.copy_(h_t, non_blocking=True)
                    else:
                        h_t.copy_(d_t, non_blocking=True)
        for i in range(n_in):
            s_c.wait_stream(s_in[i])
        e1.record(s_c)
        torch.cuda.synchronize()
        return h2d / (e0.elapsed_time(e1) * 1e-3) / 1e9

    steps = max(2, min(args.steps, args.e2e_steps))
    h2d_before = one_direction("h2d")  # the host link varies with the machine's other tenants

    def windows_of(nsets, n=5):
        for _ in range(2):
            step(nsets)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        # n timed windows of `steps` steps; the median window is reported (the host link is shared
        # with the machine's other tenants, and single windows varied by up to 1.8x)
        out = []
        for _ in range(n):
            state["computed"], state["copied_out"], state["k"] = [None, None], [None, None], 0
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_c)
            for i in range(n_in):
                s_in[i].wait_event(e0)
            for _ in range(steps):
                step(nsets)
            s_c.wait_stream(s_out)
            e1.record(s_c)
            torch.cuda.synchronize()
            out.append(max_over_ranks(e0.elapsed_time(e1), world, dev))
        return out

    windows = windows_of(2)
    ms = sorted(windows)[len(windows) // 2]
    windows1 = windows_of(1, 3)
    ms1 = sorted(windows1)[len(windows1) // 2]
    step_bytes = rs_bytes(g, S, U) + ag_bytes(U)
    value = whole_job_gbs(step_bytes, steps, world, ms)
    link = {"h2d_gbs_inputs_only_before": h2d_before, "h2d_gbs_inputs_only": one_direction("h2d"),
            "d2h_gbs_same_bytes": one_direction("d2h")}
    # a step cannot be shorter than its input copies over the host link alone, at the fastest rate
    # the link gave in this run
    h2d_ms = h2d / (max(h2d_before, link["h2d_gbs_inputs_only"]) * 1e9) * 1e3
    link["h2d_bound_ms_per_step"] = h2d_ms
    frac = h2d_ms / (ms / steps)
    # above 1 the link ran faster during the windows than when it was measured: no bound then
    link["frac_of_h2d_bound"] = frac if frac <= 1.0 else None
    if frac > 1.0:
        link["note"] = "the link measured slower than the windows ran: its rate changed during the run"
    del h_grads, h_ag, h_shards, h_params, lanes, outs, sets
    if hasattr(torch._C, "_host_emptyCache"):  # hand the 20 GB of pinned buffers back to the host
        torch._C._host_emptyCache()
    torch.cuda.empty_cache()
    return {"value": value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": ms / steps, "host_link": link,
            "windows_gbs": [whole_job_gbs(step_bytes, steps, world, w) for w in windows],
            "one_device_set": {"value": whole_job_gbs(step_bytes, steps, world, ms1), "ms_per_step": ms1 / steps,
                               "windows_gbs": [whole_job_gbs(step_bytes, steps, world, w) for w in windows1]},
            "how": "pinned host -> device copies of all inputs (4 streams), tide_reduce_scatter + "
                   "tide_all_gather, device -> pinned host copies of all outputs, every step; two device "
                   "buffer sets in turn, so step k+1's input copies overlap step k's kernels and output "
                   "copies; median of 5 windows"}


# ---- the host oracle ---------------------------------------------------------------------------


def cpu_inputs(g: Group, S: int, dev):
    """The workload's inputs as host arrays (bf16 bits): every rank's gradients and all-gather
    shards, drawn by the same seeded generator as the device buffers (on the GPU when there is one,
    then copied to the host)."""
    where = dev if (dev is not None and torch.cuda.is_available()) else "cpu"
    grads = [[rng.grad_bits(g, r, p, device=where).cpu().numpy().view(np.uint16) for p in range(g.P)]
             for r in range(g.R)]
    shards = [rng.shard_bits(g, r, S, device=where).cpu().numpy().view(np.uint16) for r in range(g.R)]
    return grads, shards


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=30).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


class HostOracle:
    """The unchanged single-threaded C oracle run over the WHOLE workload on the host's cores: one
    pass = the reduce-scatter and the all-gather placement of the full group, split into
    independent parts (one per (destination rank, parameter) and (source rank, parameter)), which
    a pool of host threads takes largest first (ctypes releases the GIL during each call, so the
    threads run in parallel).  Every part keeps the oracle's own loops and order."""

    def __init__(self, g: Group, dev=None):
        import oracle

        oracle.build()
        self.g = g
        self.lay = oracle.plan(g.R, g.rows, g.row_len)
        self.grads, self.shards = cpu_inputs(g, self.lay.S, dev)
        self.out = [np.empty(self.lay.S, np.float32) for _ in range(g.R)]
        self.params = [np.empty(g.numel(p), np.uint16) for p in range(g.P)]
        self.m_rs = oracle.marshal_reduce_scatter(self.lay, self.grads, self.out)
        self.m_ag = oracle.marshal_all_gather(self.lay, self.shards, self.params)
        rs = [("rs", d, p, int(self.lay.s[p]) * (2 * g.R + 4)) for d in range(g.R) for p in range(g.P)]
        ag = [("ag", r, p, self.lay.valid_rows(r, p) * int(self.lay.row_len[p]) * 4)
              for r in range(g.R) for p in range(g.P)]
        self.tasks = sorted(rs, key=lambda t: -t[3]) + sorted((t for t in ag if t[3]), key=lambda t: -t[3])
        self.bytes_per_pass = rs_bytes(g, self.lay.S, self.lay.U) + ag_bytes(self.lay.U)

    def _run(self, task):
        import oracle

        kind, a, p, _ = task
        if kind == "rs":
            oracle.reduce_scatter_part(self.m_rs, a, p, p + 1)
        else:
            oracle.all_gather_part(self.m_ag, a, p, p + 1)

    def time_passes(self, passes: int, warmup: int, threads: int) -> float:
        """Seconds for `passes` whole-group passes on `threads` host threads, after `warmup`.  The
        reduce-scatter parts all finish before the all-gather parts start, as in one step."""
        from concurrent.futures import ThreadPoolExecutor

        rs = [t for t in self.tasks if t[0] == "rs"]
        ag = [t for t in self.tasks if t[0] == "ag"]
        with ThreadPoolExecutor(max_workers=threads) as ex:
            def one_pass():
                list(ex.map(self._run, rs))
                list(ex.map(self._run, ag))

            for _ in range(warmup):
                one_pass()
            t0 = time.perf_counter()
            for _ in range(passes):
                one_pass()
            return time.perf_counter() - t0


def host_threads() -> int:
    return len(os.sched_getaffinity(0))


def cpu_baseline(g: Group, dev, passes: int = 3) -> dict:
    """The oracle as it stands, on every host core this process may use, over the whole workload
    (the reduce-scatter and the placement of the full group, the same bytes as one GPU step); and
    one pass on a single thread for scale."""
    ho = HostOracle(g, dev)
    n = host_threads()
    dt = ho.time_passes(passes, 1, n)
    dt1 = ho.time_passes(1, 0, 1)
    res = {"value": ho.bytes_per_pass * passes / dt / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
           "seconds": dt, "passes": passes,
           "sample": f"the whole {g.name} group (R = {g.R}, P = {g.P}): reduce-scatter + all-gather placement, "
                     f"{ho.bytes_per_pass / 1e9:.2f} GB of algorithmic traffic per pass, {passes} passes after 1 "
                     f"warm-up, {n} host threads over (rank, parameter) parts of the single-threaded C oracle",
           "one_thread_gbs": ho.bytes_per_pass / dt1 / 1e9,
           "host_cpus": os.cpu_count(), "cpu_model": cpu_model()}
    del ho
    return res


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands (single-threaded C loops), over the same
    workload as the GPU arm, on all the host cores this process may use (threads over (rank,
    parameter) parts).  A step = one reduce-scatter + all-gather placement of the whole group."""
    g = workload(args)
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    ho = HostOracle(g, dev)
    n = host_threads()
    dt = ho.time_passes(args.steps, args.warmup, n)
    value = ho.bytes_per_pass * args.steps / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": DATA,
        "config": workload_config(g, ho.lay.S, ho.lay.U, 1),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle",
                         "sample": f"the whole {g.name} group per step (no sampling), {n} host threads over "
                                   f"(rank, parameter) parts of the single-threaded C oracle",
                         "cpu_model": cpu_model(), "host_cpus": os.cpu_count()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["tide", "reference"], default="tide")
    ap.add_argument("--workload", default="llama70b")
    ap.add_argument("--scale", type=int, default=1, help="divide every dimension by this (profiling cases)")
    ap.add_argument("--rs-ctas", type=int, default=0)
    ap.add_argument("--ag-ctas", type=int, default=0)
    ap.add_argument("--rs-variant", choices=["auto", "register", "bulk", "tmem"], default="auto")
    ap.add_argument("--ag-variant", choices=["auto", "register", "bulk"], default="auto")
    ap.add_argument("--ce-lanes", type=int, default=0, help="copy-engine streams (0 = library default)")
    ap.add_argument("--ce-lanes-sweep", type=int, nargs="*", default=[])
    ap.add_argument("--ce-bands-sweep", type=int, nargs="*", default=[2, 4, 8])
    ap.add_argument("--interference-ctas", type=int, nargs="*", default=[8, 12, 16, 20, 24, 32])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-passes", type=int, default=3, help="whole-group oracle passes of the CPU baseline")
    ap.add_argument("--sweep", action="store_true", help="CTA-count sweep of bandwidth vs GEMM slowdown")
    ap.add_argument("--sweep-rs", type=int, nargs="*", default=[8, 16, 20, 24, 32, 48, 64, 96, 152, 304])
    ap.add_argument("--sweep-ag", type=int, nargs="*", default=[8, 16, 24, 32, 64, 152, 608])
    ap.add_argument("--probes", action="store_true", help="spin-CTA curve, SM-id probe and Table 4 victims")
    ap.add_argument("--slot-reuse", action="store_true", help="Slot-Reuse staging leg")
    ap.add_argument("--overlap-ce-forms", action="store_true",
                    help="copy-engine placement over one lane in both forms beside the GEMM")
    ap.add_argument("--spin-ctas", type=int, nargs="*", default=[1, 4, 8, 12, 16, 20, 24, 32, 48, 64, 96, 152])
    ap.add_argument("--no-interference", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-stock", action="store_true", help="skip the one-GPU pack/copy-out comparator")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from all_gather_tide_gb300 import build as _b

    if not os.path.exists(_b.LIB):
        raise SystemExit(f"{_b.LIB} is missing: run __graft_entry__.build() first")
    out = run_tide(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

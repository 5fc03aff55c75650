"""Builds ``libtide.so`` in-tree with nvcc for sm_103a (translation units compiled in parallel).

    python -m all_gather_tide_gb300.build [--force] [--ptxas-verbose]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtide.so")
SOURCES = ["plan.cpp", "tide_api.cpp", "rs_kernel.cu", "rs_bulk_kernel.cu", "ag_kernel.cu", "ag_bulk_kernel.cu", "noalloc.cu", "probes.cu"]
HEADERS = [os.path.join(CSRC, "tide_internal.h"), os.path.join(ROOT, "include", "tide.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def _flags(ptxas_verbose: bool):
    f = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    nv = nvcc()
    os.makedirs(BUILD, exist_ok=True)
    objs = []
    jobs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if force or ptxas_verbose or _stale(obj, [path, *HEADERS]):
            x = ["-x", "cu"] if src.endswith(".cu") else ["-x", "c++"]
            jobs.append([nv, *_flags(ptxas_verbose), *x, "-c", path, "-o", obj])

    def run(cmd):
        return subprocess.run(cmd, capture_output=True, text=True)

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, res in zip(jobs, ex.map(run, jobs)):
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
            if not quiet or ptxas_verbose:
                sys.stdout.write(res.stdout + res.stderr)
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        libdir = cuda_lib_dir(nv)
        cmd = [nv, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "shared",
               "-Xlinker", f"-rpath,{libdir}", "-L", libdir]
        res = run(cmd)
        if res.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose, quiet=False))

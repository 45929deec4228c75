"""Build the CUDA libraries in-tree with nvcc for sm_103a.

    libwsattn.so         the product: C ABI of include/wsattn.h (+ wsattn_testing.h)
    libwsattn_probes.so  test-only single-tile kernels (include/wsattn_probes.h)

Translation units compile in parallel; ptxas resource usage (registers,
spills, shared memory) is kept in _build/ptxas_<unit>.txt.
Run: python -m warp_specialized_attention_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libwsattn.so")
PROBES = os.path.join(PKG, "libwsattn_probes.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I" + INCLUDE, "-I" + CSRC]

LIB_UNITS = ["fmha_api.cu", "fmha_fwd_d64.cu", "fmha_fwd_d128.cu", "fmha_fwd_e4m3.cu",
             "fmha_fwd_ksplit.cu", "fmha_bwd.cu"]
PROBE_UNITS = ["probes.cu"]
HEADERS = ["ptx.cuh", "fmha_fwd_sm103.cuh", "fmha_bwd_sm103.cuh", "fmha_launch.h"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libwsattn")


def _inputs(units):
    paths = [os.path.join(CSRC, u) for u in units] + [os.path.join(CSRC, h) for h in HEADERS]
    paths += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return paths


def _stale(target, units) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(p) > t for p in _inputs(units))


def _compile(unit: str) -> str:
    src = os.path.join(CSRC, unit)
    obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
    r = subprocess.run([_nvcc(), *ARCH, *FLAGS, "-c", src, "-o", obj],
                       capture_output=True, text=True)
    with open(os.path.join(BUILD, "ptxas_" + unit.replace(".cu", ".txt")), "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (unit, r.stderr[-6000:]))
    return obj


def _link(objs, target):
    tmp = target + ".tmp.%d" % os.getpid()
    r = subprocess.run([_nvcc(), *ARCH, "-shared", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link of %s failed:\n%s" % (target, r.stderr[-4000:]))
    os.replace(tmp, target)


def build(force: bool = False, probes: bool = True) -> str:
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    if force or _stale(LIB, LIB_UNITS):
        jobs.append((LIB, LIB_UNITS))
    if probes and (force or _stale(PROBES, PROBE_UNITS)):
        jobs.append((PROBES, PROBE_UNITS))
    units = [u for _, us in jobs for u in us]
    if units:
        with cf.ThreadPoolExecutor(max_workers=min(len(units), os.cpu_count() or 4)) as ex:
            objs = dict(zip(units, ex.map(_compile, units)))
        for target, us in jobs:
            _link([objs[u] for u in us], target)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv)
    print(LIB)

"""Build libmoe.so from csrc/ with nvcc for sm_103a (no cmake, no torch).

Each translation unit is compiled in parallel into ``_build/``; the shared
library is linked next to this file, where the binding loads it from.

Variants (``python -m combine_moe_layout_02_gb300.build --variant NAME``) are
the same sources compiled with extra defines into ``libmoe_NAME.so``; the
binding loads one when ``MOE_LIBRARY=NAME`` is set:
  match_hist   layout's histograms in the atomics-free grouped form
               (-DMOE_LAYOUT_MATCH_HIST) instead of shared-memory atomics
  profile      kernels record per-CTA phase times into a device array
               attached with moe_profile_attach (-DMOE_PROFILE)
"""

from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libmoe.so")
SOURCES = ["api.cu", "layout.cu", "notify.cu", "dispatch.cu", "combine.cu", "layout_static.cu", "pad.cu", "expert.cu", "fused.cu", "run.cu", "exchange.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
VARIANTS = {"match_hist": ["-DMOE_LAYOUT_MATCH_HIST"], "profile": ["-DMOE_PROFILE"]}


def lib_path(variant: str | None = None) -> str:
    return LIB if not variant else os.path.join(HERE, f"libmoe_{variant}.so")


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
            "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *extra]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, variant: str | None = None) -> str:
    defines = VARIANTS[variant] if variant else []
    out_dir = os.path.join(BUILD, variant) if variant else BUILD
    lib = lib_path(variant)
    os.makedirs(out_dir, exist_ok=True)
    # Objects built on another host architecture are never reused.
    stamp = os.path.join(out_dir, "HOST")
    host = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != host:
        force = True
    headers = [os.path.join(INCLUDE, "moe.h"), os.path.join(CSRC, "moe_device.cuh")]
    cc = nvcc()
    jobs = []
    objs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or ptxas_info or _stale(obj, [path, *headers]):
            extra = (["-Xptxas", "-v"] if ptxas_info else []) + defines
            jobs.append([cc, *_flags(extra), "-c", path, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_info or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    with open(stamp, "w") as f:
        f.write(host + "\n")
    if force or jobs or _stale(lib, objs) or not os.path.exists(lib):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    var = sys.argv[sys.argv.index("--variant") + 1] if "--variant" in sys.argv else None
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv, variant=var))

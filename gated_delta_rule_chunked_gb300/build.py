"""Build libkda.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into one shared
library next to this file. Set KDA_PTXAS_VERBOSE=1 to print register and
shared-memory usage per kernel.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkda.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["kda_api.cu", "kda_step.cu", "kda_prep.cu", "kda_prep_tc.cu", "kda_scan.cu", "kda_scan_tc.cu", "kda_bwd_tc.cu", "kda_bwd_f32.cu", "kda_conv.cu",
           "kda_cp.cu", "kda_attnres.cu", "kda_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags():
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if os.environ.get("KDA_PTXAS_VERBOSE"):
        f += ["-Xptxas", "-v"]
    return f


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "kda.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s.replace(".cu", ".o"))
        if force or _stale(obj, src):
            jobs.append((src, obj))

    def run(job):
        src, obj = job
        cmd = [cc] + _flags() + ["-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for log in ex.map(run, jobs):
            if verbose and log:
                sys.stderr.write(log)
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([cc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

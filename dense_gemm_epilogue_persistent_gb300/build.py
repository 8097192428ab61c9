"""Compile the CUDA library ``libgemm_gb300.so`` in-tree for sm_103a.

The translation units are compiled in parallel with nvcc
(``-gencode arch=compute_103a,code=sm_103a -lineinfo``) and linked into one
shared object next to this file; the CUDA runtime is linked statically, so
loading the library needs no GPU and no libcuda (the driver's tensor-map
encoder is resolved through the runtime at ``gemm_create`` time).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "gemm_gb300")
LIB = os.path.join(HERE, "libgemm_gb300.so")
# The ring-statistics build: the same sources with per-role wait counters
# compiled in (GB300_RING_STATS=1), a separate library for studying the
# pipeline; the product library compiles none of it.
STATS_BUILD = os.path.join(ROOT, "_build", "gemm_gb300_stats")
STATS_LIB = os.path.join(HERE, "libgemm_gb300_stats.so")

SOURCES = ["gemm_api.cu", "kern_ab16_mc1.cu", "kern_ab16_mc2.cu", "kern_ab8_mc1.cu",
           "kern_ab8_mc2.cu", "kern_ab32_mc1.cu", "kern_ab32_mc2.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
         "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgemm_gb300.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gemm_gb300.h"))
    return files


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ring_stats: bool = False) -> str:
    """Build the library if any source is newer than it; return its path.
    ring_stats: build the ring-statistics library instead of the product one."""
    lib = STATS_LIB if ring_stats else LIB
    bdir = STATS_BUILD if ring_stats else BUILD
    extra = ["-DGB300_RING_STATS=1"] if ring_stats else []
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(bdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ring_stats="--ring-stats" in sys.argv))

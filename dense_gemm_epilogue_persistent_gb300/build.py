"""Compile the CUDA libraries in-tree for sm_103a.

Four libraries are built from the sources in ``csrc/`` (nvcc,
``-gencode arch=compute_103a,code=sm_103a -lineinfo``, translation units in
parallel, the CUDA runtime linked statically so that loading a library needs
neither a GPU nor libcuda):

``libgemm_gb300.so``       the library for a process that drives one GPU: every
                           kernel variant, including the clusters whose CTAs
                           share operand tiles through TMA multicast.
``libgemm_gb300_nomc.so``  the library for processes that drive several GPUs:
                           built only from translation units and headers that
                           contain no multicast TMA load (kern_shared.cu and
                           ptx_multicast.cuh are left out, and the host code
                           is compiled with GB300_MULTICAST=0, so a forced
                           multicast cluster returns
                           GEMM_ERR_UNSUPPORTED_CONFIG).
``libgemm_gb300_stats.so`` the ring-statistics build (GB300_RING_STATS=1):
                           the single-GPU library with per-role wait counters,
                           for studying the pipeline; built only on request.
``libgemm_gb300_debug.so`` the debug build (GB300_DEBUG=1): the single-GPU
                           library with device-side bounds checks of every TMA
                           box, store coordinate and tensor-memory column
                           range, reported as GEMM_ERR_DEVICE_CHECK; built
                           only on request.

Each kernel unit is compiled once per input width (and per epilogue warp
count and stream-K form for kern_plain.cu, per cluster shape for
kern_shared.cu) with -D flags, so the units compile in parallel.
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
BUILD_ROOT = os.path.join(ROOT, "_build")

LIBS = {
    "product": os.path.join(HERE, "libgemm_gb300.so"),
    "nomc": os.path.join(HERE, "libgemm_gb300_nomc.so"),
    "stats": os.path.join(HERE, "libgemm_gb300_stats.so"),
    "debug": os.path.join(HERE, "libgemm_gb300_debug.so"),
}
LIB = LIBS["product"]
NOMC_LIB = LIBS["nomc"]
STATS_LIB = LIBS["stats"]
DEBUG_LIB = LIBS["debug"]
EXTRA_DEFINES = {"stats": ["-DGB300_RING_STATS=1"], "debug": ["-DGB300_DEBUG=1"]}

# (object name, source, -D flags).  Input widths: 2 bytes (fp16/bf16), 1 (fp8),
# 4 (tf32); epilogue warps per tensor-memory lane quarter (1 or 2); stream-K
# items or not; operand-sharing cluster shapes (groups along M, along N).
PLAIN_UNITS = [(f"kern_plain_ab{ab}_e{epw}_s{sk}", "kern_plain.cu",
                [f"-DGB300_AB={ab}", f"-DGB300_EPW={epw}", f"-DGB300_SK={sk}"])
               for ab in (2, 1, 4) for epw in (1, 2) for sk in (0, 1)]
SHARED_UNITS = [(f"kern_shared_ab{ab}_m{mc}_n{nc}", "kern_shared.cu",
                 [f"-DGB300_AB={ab}", f"-DGB300_MC={mc}", f"-DGB300_NC={nc}"])
                for ab in (2, 1, 4) for mc, nc in ((2, 1), (1, 2), (2, 2))]
# Files the multi-GPU library is built from (its translation units and every
# header they include): none of them names a multicast TMA load.
NOMC_FILES = ["gemm_api.cu", "kern_plain.cu", "gemm_kernel.cuh", "ptx.cuh", "kernels.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
         "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def units(kind: str):
    """Translation units of one library: (object name, source, -D flags)."""
    if kind == "nomc":
        return [("gemm_api_nomc", "gemm_api.cu", ["-DGB300_MULTICAST=0"])] + PLAIN_UNITS
    return [("gemm_api", "gemm_api.cu", ["-DGB300_MULTICAST=1"])] + PLAIN_UNITS + SHARED_UNITS


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the GEMM library")


def _inputs(kind: str):
    names = NOMC_FILES if kind == "nomc" else os.listdir(CSRC)
    files = [os.path.join(CSRC, f) for f in names]
    files.append(os.path.join(INCLUDE, "gemm_gb300.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib: str, kind: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs(kind))


def build(force: bool = False, verbose: bool = False, ring_stats: bool = False,
          kind: str | None = None) -> str:
    """Build one library if any of its sources is newer than it; return its
    path.  kind: "product" (default), "nomc", "stats" or "debug" (ring_stats=True
    is the same as kind="stats")."""
    kind = kind or ("stats" if ring_stats else "product")
    lib = LIBS[kind]
    if not force and not _stale(lib, kind):
        return lib
    nvcc = _nvcc()
    bdir = os.path.join(BUILD_ROOT, f"gemm_gb300_{kind}")
    os.makedirs(bdir, exist_ok=True)
    extra = EXTRA_DEFINES.get(kind, [])

    def compile_one(unit):
        name, src, defs = unit
        obj = os.path.join(bdir, name + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defs, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} {defs}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(f"== {name}\n{r.stderr}")
        return obj

    us = units(kind)
    with cf.ThreadPoolExecutor(min(len(us), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, us))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    k = next((v for f, v in (("--ring-stats", "stats"), ("--nomc", "nomc"), ("--debug", "debug"))
              if f in sys.argv), "product")
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, kind=k))

"""The library for processes that drive several GPUs (no multicast kernels),
run in a subprocess so that the test process keeps the single-GPU library:
plain clusters compute the same results as the single-GPU library within the
parity bound, and a forced multicast cluster is refused with
GEMM_ERR_UNSUPPORTED_CONFIG."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, "tests")
import dense_gemm_epilogue_persistent_gb300 as G
from dense_gemm_epilogue_persistent_gb300 import build as B
G.select_library(B.build(kind="nomc"))
from gemm_cases import Case, compare_full, prepare, run_gpu
g = G.Gemm(0)
cases = [Case(M=700, N=520, K=264, L=2, ab="f16", c="f16", d="f16", x="f16", y="f16",
              alpha=2.0, beta=1.0, xf=3.0, seed=5),
         Case(M=300, N=504, K=272, L=1, ab="e4m3", c="f16", d="f16", alpha=0.25, beta=1.0,
              dist="e4m3_pm4", seed=4)]
for case in cases:
    for cfg in (None, dict(cta_group=2, tile_n=192), dict(cta_group=1, tile_n=128)):
        g.set_config(**cfg) if cfg else g.set_config(None)
        prep = prepare(case)
        D, Y = run_gpu(g, prep)
        st, detail = g.sync_status()
        assert st == G.GEMM_OK, (st, hex(detail))
        compare_full(prep, D, Y)
        c = g.last_config()
        assert (c.cluster_m, c.cluster_n) == (1, 1)
for cm, cn in ((2, 1), (1, 2), (2, 2)):
    g.set_config(cluster_m=cm, cluster_n=cn)
    try:
        run_gpu(g, prepare(cases[0]))
        raise SystemExit("multicast cluster ran in the multi-GPU library")
    except G.GemmError as e:
        assert e.status == G.GEMM_ERR_UNSUPPORTED_CONFIG, e
g.close()
import ctypes
maps = open("/proc/self/maps").read()
assert "libgemm_gb300_nomc.so" in maps and "libgemm_gb300.so" not in maps
print("NOMC_OK")
'''


def test_multi_gpu_library_runs_plain_clusters_and_refuses_multicast():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "NOMC_OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]

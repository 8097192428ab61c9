"""The debug library (GB300_DEBUG=1: device-side bounds checks of every TMA
box, TMA store coordinate and tensor-memory column range, recorded in the
status word instead of trapping), built here from the same sources and run
in a subprocess so that the test process keeps the product library: on
ragged problems across tile widths, cluster shapes, MN-major operands, the
split last wave and K = 0 no check fires and the results stay within the
parity bound of the oracle."""
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
G.select_library(B.build(kind="debug"))
from gemm_cases import Case, compare_full, prepare, run_gpu
g = G.Gemm(0)
cases = [
    (Case(M=720, N=704, K=400, L=2, ab="bf16", c="f16", d="f32", x="bf16", y="f16",
          a_mn=True, b_mn=True, alpha=-0.75, beta=1.0, xf=0.5, seed=31),
     [None, (2, 256, 1, 2), (2, 256, 2, 2), (1, 128, 2, 1), (2, 128, 1, 1), (1, 64, 1, 1),
      (2, 256, 1, 1, 2), (1, 192, 1, 1, 2), (1, 256, 1, 1, 2, 2), (2, 128, 1, 1, 1, 2)]),
    (Case(M=300, N=504, K=272, L=1, ab="e4m3", c="f16", d="f16", alpha=0.25, beta=1.0,
          dist="e4m3_pm4", seed=4),
     [None, (2, 224, 1, 1), (1, 160, 1, 1), (2, 96, 2, 1), (2, 192, 1, 1)]),
    (Case(M=2560, N=1920, K=192, L=1, ab="f16", c="f16", d="f16", x="bf16", y="f16",
          alpha=1.0, beta=-0.5, xf=2.0, seed=77),                 # split last wave
     [(2, 192, 1, 1), (2, 256, 1, 1), (2, 192, 1, 1, 2)]),
    (Case(M=200, N=136, K=0, L=2, ab="bf16", c="f32", d="f32", x="f16", y="f32",
          alpha=1.0, beta=0.5, xf=2.0, seed=8), [None]),
    (Case(M=264, N=320, K=200, L=3, ab="bf16", c="bf16", d="bf16", a_mn=True, b_mn=True,
          cd_m=True, alpha=0.5, beta=0.0, dist="normal002", seed=3), [None, (1, 256, 1, 1)]),
]
n = 0
for case, variants in cases:
    for v in variants:
        if v:
            g.set_config(cta_group=v[0], tile_n=v[1], cluster_m=v[2], cluster_n=v[3],
                         epi_warps=v[4] if len(v) > 4 else 0,
                         stream_k=v[5] if len(v) > 5 else 0)
        else:
            g.set_config(None)
        prep = prepare(case)
        D, Y = run_gpu(g, prep)
        st, detail = g.sync_status()
        assert st == G.GEMM_OK, (G.gemm_status_string(st), hex(detail), v)
        compare_full(prep, D, Y)
        n += 1
g.close()
maps = open("/proc/self/maps").read()
assert "libgemm_gb300_debug.so" in maps
print("DEBUG_OK", n)
'''


def test_debug_build_checks_pass_on_valid_problems():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0 and "DEBUG_OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]

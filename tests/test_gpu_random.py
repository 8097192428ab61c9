"""Randomised GPU parity: 80 seeded problems drawn across every input type, accumulator,
layout, optional tensor, epilogue variant, kernel variant and ragged shape the library
takes, each compared element by element with the fp64 oracle (the bounds of
gemm_cases).  Shapes keep the leading dimensions 16-byte aligned, as the C ABI
requires, and the work small enough for the oracle to finish in seconds."""
import numpy as np
import pytest
import torch

import dense_gemm_epilogue_persistent_gb300 as G
import workloads as W
from gemm_cases import Case, compare_full, prepare, run_gpu

pytestmark = pytest.mark.gpu

AB = [("f16", None), ("bf16", None), ("e4m3", None), ("e5m2", None), ("e4m3", "e5m2"),
      ("e5m2", "e4m3"), ("tf32", None)]
OUT = ["f32", "f16", "bf16"]
# (cta_group, tile_n, cluster_m, cluster_n[, epi_warps]), None = automatic
VARIANTS = [None, (1, 128, 1, 1), (1, 256, 1, 1), (2, 128, 1, 1), (2, 256, 1, 1),
            (1, 128, 2, 1), (1, 256, 2, 1), (2, 128, 2, 1), (2, 256, 2, 1),
            (1, 64, 1, 1), (1, 96, 1, 1), (1, 160, 1, 1), (1, 192, 1, 1), (1, 224, 1, 1),
            (2, 64, 1, 1), (2, 96, 1, 1), (2, 160, 1, 1), (2, 192, 1, 1), (2, 224, 1, 1),
            (1, 128, 1, 2), (2, 256, 1, 2), (2, 160, 1, 2), (1, 96, 2, 2), (2, 224, 2, 2),
            (1, 128, 1, 1, 2), (2, 256, 1, 1, 2), (1, 96, 1, 1, 2), (2, 192, 1, 1, 2)]
N_CASES = 80


def _round_up(v, m):
    return (v + m - 1) // m * m


def draw_case(i):
    """Case i of the seeded stream (pure host logic, no GPU)."""
    g = np.random.default_rng(7000 + i)
    ab, b = AB[g.integers(len(AB))]
    es = W.ELEM_BYTES[ab]
    tf32 = ab == "tf32"
    a_mn = bool(g.integers(2)) and not tf32
    b_mn = bool(g.integers(2)) and not tf32
    cd_m = bool(g.integers(2))
    c = OUT[g.integers(3)] if g.random() < 0.8 else None
    d = OUT[g.integers(3)]
    x = OUT[g.integers(3)] if g.random() < 0.5 else None
    y = OUT[g.integers(3)] if g.random() < 0.5 else None
    acc = "f16" if (ab in ("f16", "e4m3", "e5m2") and g.random() < 0.3) else "f32"
    # 16-byte rows: K (K-major operands), M / N (MN-major operands and the
    # C/D/X/Y leading dimension) rounded to what every involved type needs
    k_mult = 16 // es
    mn_mult = 16 // es
    out_mult = 8 if any(t in ("f16", "bf16") for t in (c, d, x, y) if t) else 4
    M = int(g.integers(1, 700))
    N = int(g.integers(1, 700))
    K = int(g.integers(1, 520))
    L = int(g.integers(1, 4))
    K = _round_up(K, k_mult)
    if a_mn:
        M = _round_up(M, mn_mult)
    if b_mn:
        N = _round_up(N, mn_mult)
    if cd_m:
        M = _round_up(M, out_mult)
    else:
        N = _round_up(N, out_mult)
    if acc == "f16":
        K = min(K, 256)              # keep |running sums| well inside fp16's range
    scal = lambda: float(g.choice([-2.0, -1.0, -0.5, 0.0, 0.25, 0.5, 1.0, 1.5, 3.0]))
    alpha = scal() or 1.0
    beta = scal() if c else 0.0
    xf = scal() if x else 0.0
    relu = bool(g.random() < 0.3)
    dist = "e4m3_pm4" if ab in ("e4m3", "e5m2") else ("normal1" if g.random() < 0.7 else "uniform1")
    variant = VARIANTS[g.integers(len(VARIANTS))]
    case = Case(M=M, N=N, K=K, L=L, ab=ab, b=b, c=c, d=d, x=x, y=y, a_mn=a_mn, b_mn=b_mn,
                cd_m=cd_m, alpha=alpha, beta=beta, xf=xf, dist=dist, seed=9000 + i, relu=relu,
                acc=acc)
    return case, variant


@pytest.fixture(scope="module")
def gemm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    h = G.Gemm(0)
    yield h
    h.close()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_problem(gemm, i):
    case, variant = draw_case(i)
    if variant:
        cg, bn, mc, nc = variant[:4]
        epw = variant[4] if len(variant) > 4 else 0
        gemm.set_config(cta_group=cg, tile_n=bn, cluster_m=mc, cluster_n=nc, epi_warps=epw)
    else:
        gemm.set_config(None)
    prep = prepare(case)
    try:
        D, Y = run_gpu(gemm, prep)
    except G.GemmError as ex:
        # a forced variant may not fit the problem (e.g. a cluster of CTA pairs
        # on a tiny M); the automatic choice must always run it
        assert ex.status == G.GEMM_ERR_UNSUPPORTED_CONFIG and variant, ex
        gemm.set_config(None)
        D, Y = run_gpu(gemm, prep)
    st, detail = gemm.sync_status()
    assert st == G.GEMM_OK, f"{G.gemm_status_string(st)} {detail:#x}"
    compare_full(prep, D, Y)
    gemm.set_config(None)

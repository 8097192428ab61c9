"""gemm_run_noalloc: the GEMM entry point for callers that must not allocate
device memory (a framework pool that owns the GPU's memory, latency-critical
loops that cannot afford cudaMalloc's device-wide synchronisation, or rules
that forbid allocation after start-up).  Its one piece of scratch, the
kernel's watchdog status word, sits in a static device array instead of
memory gemm_create would allocate.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It must also pass alone in a
fresh process, where its first call performs the per-device set-up; the last
test here runs the others that way.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads as W
import dense_gemm_epilogue_persistent_gb300 as G
from gemm_cases import Case, assert_within, bound_D, logical, oracle_problem, out_shape, prepare, \
    TOL_REL, to_f64, ulp_at
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # custom epilogue, ragged, several tiles per cluster
    Case(M=1100, N=776, K=520, L=2, ab="f16", c="f16", d="f16", x="f16", y="f16", alpha=2.0,
         beta=1.0, xf=3.0, seed=101),
    # batched, M-major A / N-major B / M-major C and D, fp32 output
    Case(M=520, N=384, K=264, L=3, ab="bf16", c="bf16", d="f32", a_mn=True, b_mn=True,
         cd_m=True, alpha=0.5, beta=-1.0, seed=102),
]


def _device_inputs(prep):
    dev = torch.device("cuda")
    A, B = prep.A.to(dev), prep.B.to(dev)
    C = prep.C.to(dev) if prep.C is not None else None
    X = prep.X.to(dev) if prep.X is not None else None
    return A, B, C, X


def _outputs(case):
    D = torch.full(out_shape(case), float("nan"), dtype=W.TORCH_DTYPE[case.d], device="cuda")
    Y = (torch.full(out_shape(case), float("nan"), dtype=W.TORCH_DTYPE[case.y], device="cuda")
         if case.y else None)
    return D, Y


def _dtypes(case):
    return G.make_dtypes(case.ab, case.c or "f32", case.d, case.x or "f32", case.y or "f32",
                         G.GEMM_MN_MAJOR if case.cd_m else G.GEMM_K_MAJOR)


def _run_handle(g, prep, stream):
    c = prep.case
    A, B, C, X = _device_inputs(prep)
    D, Y = _outputs(c)
    g.run(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B, B.shape[-1], int(c.b_mn), C, X,
          D, Y, c.alpha, c.beta, c.xf, _dtypes(c), stream)
    st, detail = g.sync_status(stream)
    assert st == G.GEMM_OK, (G.gemm_status_string(st), hex(detail))
    return D, Y


def test_handle_still_runs_after_noalloc():
    """A handle whose launch was prepared (with the most shared memory its
    kernel allows) before the first no-allocation call must still launch
    afterwards: the one-time set-up of gemm_run_noalloc may raise, but never
    lower, a kernel's process-wide shared-memory limit.  Runs first in this
    file, so in a fresh process the set-up happens between the two launches."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    prep = prepare(CASES[0])
    stream = torch.cuda.current_stream()
    g = G.Gemm(0)
    try:
        g.set_config(cta_group=2, tile_n=256, cluster_m=2)
        D0, Y0 = _run_handle(g, prep, stream)
        c = prep.case
        A, B, C, X = _device_inputs(prep)
        D1, Y1 = _outputs(c)
        st, word = G.gemm_run_noalloc(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B,
                                      B.shape[-1], int(c.b_mn), C, X, D1, Y1, c.alpha, c.beta,
                                      c.xf, _dtypes(c), stream, watchdog=True)
        assert st == G.GEMM_OK and word == 0
        D2, Y2 = _run_handle(g, prep, stream)     # the cached launch, after the set-up
        assert torch.equal(D0, D2) and torch.equal(Y0, Y2)
    finally:
        g.close()


def test_noalloc_matches_gemm_run_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    preps = [prepare(c) for c in CASES]
    # two no-allocation calls back to back on one stream (the second reuses
    # the scratch the first left behind)...
    stream = torch.cuda.current_stream()
    got = []
    for prep in preps:
        c = prep.case
        A, B, C, X = _device_inputs(prep)
        D, Y = _outputs(c)
        st, _ = G.gemm_run_noalloc(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B,
                                   B.shape[-1], int(c.b_mn), C, X, D, Y, c.alpha, c.beta, c.xf,
                                   _dtypes(c), stream)
        assert st == G.GEMM_OK
        got.append((D, Y, (A, B, C, X)))
    # ...then a synchronising call that reports the watchdog word
    c = preps[0].case
    A, B, C, X = got[0][2]
    D_sync, Y_sync = _outputs(c)
    st, word = G.gemm_run_noalloc(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B,
                                  B.shape[-1], int(c.b_mn), C, X, D_sync, Y_sync, c.alpha,
                                  c.beta, c.xf, _dtypes(c), stream, watchdog=True)
    assert st == G.GEMM_OK and word == 0
    torch.cuda.synchronize()

    # a warm call allocates nothing: neither device memory (free bytes of the
    # device) nor anything from torch's caching allocator
    free0 = torch.cuda.mem_get_info()[0]
    n_alloc0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    st, word = G.gemm_run_noalloc(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B,
                                  B.shape[-1], int(c.b_mn), C, X, D_sync, Y_sync, c.alpha,
                                  c.beta, c.xf, _dtypes(c), stream, watchdog=True)
    assert st == G.GEMM_OK and word == 0
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == n_alloc0

    # the same problems through the existing entry point
    g = G.Gemm(0)
    try:
        for prep, (D, Y, (A, B, C, X)) in zip(preps, got):
            c = prep.case
            D_ref, Y_ref = _outputs(c)
            g.run(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B, B.shape[-1], int(c.b_mn),
                  C, X, D_ref, Y_ref, c.alpha, c.beta, c.xf, _dtypes(c), stream)
            st, detail = g.sync_status(stream)
            assert st == G.GEMM_OK, detail
            # within the parity bound the other tests use (scaled by the
            # oracle's sum |a*b| for these inputs)
            D_exact, Y_exact, S = oracle.gemm(oracle_problem(prep))
            Cv = to_f64(prep.inp.C) if prep.inp.C is not None else None
            Xv = to_f64(prep.inp.X) if prep.inp.X is not None else None
            d_new = to_f64(logical(D, c.cd_m))
            d_old = to_f64(logical(D_ref, c.cd_m))
            assert_within("D noalloc vs gemm_run", d_new, d_old, bound_D(c, S, Cv, Xv, D_exact))
            assert_within("D noalloc vs oracle", d_new, D_exact, bound_D(c, S, Cv, Xv, D_exact))
            if Y is not None:
                y_new = to_f64(logical(Y, c.cd_m))
                y_old = to_f64(logical(Y_ref, c.cd_m))
                assert_within("Y noalloc vs gemm_run", y_new, y_old,
                              TOL_REL * S + ulp_at(c.y, Y_exact))
                assert_within("Y noalloc vs oracle", y_new, Y_exact,
                              TOL_REL * S + ulp_at(c.y, Y_exact))
        # the synchronising call gave the same result as the first call
        assert torch.equal(D_sync, got[0][0]) and torch.equal(Y_sync, got[0][1])
    finally:
        g.close()


def test_noalloc_alone_in_a_fresh_process():
    """The tests above, run again in a new process where nothing else has
    touched the library: the first no-allocation call does the set-up."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if os.environ.get("GEMM_NOALLOC_CHILD"):
        pytest.skip("already the fresh process")
    env = dict(os.environ, GEMM_NOALLOC_CHILD="1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.abspath(__file__), "-k", "not fresh_process"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "2 passed" in r.stdout, r.stdout[-2000:]

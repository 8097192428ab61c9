"""GPU parity at the largest extents the tests can afford.

Outputs of more than 2^31 elements (row-major, and column-major with a batch
that starts beyond 2^31 bytes) check that every offset the kernel and its
tensor maps form is 64-bit; a K of 2^20 runs 8192 ring stages through one
accumulator.  All inputs are small integers, so every product and partial sum
is exact in fp32 and the outputs must equal the once-rounded oracle bit for
bit.  Entries are gathered on the device (random ones, the first and last
rows and columns, the last element) and computed one by one by the oracle;
guard elements after each output must stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import dense_gemm_epilogue_persistent_gb300 as G
from gemm_cases import Case, oracle_problem, prepare

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements after each output that must keep their sentinel


@pytest.fixture(scope="module")
def gemm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g = G.Gemm(0)
    yield g
    g.close()


def _guarded(shape, dtype, dev):
    n = int(np.prod(shape))
    flat = torch.full((n + GUARD,), 7.0, dtype=dtype, device=dev)
    return flat, flat[:n].view(shape)


def _entries(M, N, L, seed, n_random):
    rng = np.random.default_rng(seed)
    ms = [rng.integers(0, M, n_random)]
    ns = [rng.integers(0, N, n_random)]
    ls = [rng.integers(0, L, n_random)]
    for l in sorted({0, L - 1}):
        for r in (0, M - 1):
            ms.append(np.full(N, r)); ns.append(np.arange(N)); ls.append(np.full(N, l))
        for c in (0, N - 1):
            ms.append(np.arange(M)); ns.append(np.full(M, c)); ls.append(np.full(M, l))
    ms.append(np.array([M - 1])); ns.append(np.array([N - 1])); ls.append(np.array([L - 1]))
    return np.concatenate(ms), np.concatenate(ns), np.concatenate(ls)


def _run_exact(gemm, case, n_random=2048):
    prep = prepare(case)
    dev = torch.device("cuda")
    A = prep.A.to(dev)
    B = prep.B.to(dev)
    C = prep.C.to(dev) if prep.C is not None else None
    shape = (case.L, case.N, case.M) if case.cd_m else (case.L, case.M, case.N)
    dflat, D = _guarded(shape, W.TORCH_DTYPE[case.d], dev)
    dt = G.make_dtypes(case.ab, case.c or "f32", case.d, "f32", "f32",
                       G.GEMM_MN_MAJOR if case.cd_m else G.GEMM_K_MAJOR)
    gemm.run(case.M, case.N, case.K, case.L, A, A.shape[-1], int(case.a_mn), B, B.shape[-1],
             int(case.b_mn), C, None, D, None, case.alpha, case.beta, 0.0, dt, None)
    st, detail = gemm.sync_status()
    assert st == G.GEMM_OK, f"{G.gemm_status_string(st)} {detail:#x}"
    ms, ns, ls = _entries(case.M, case.N, case.L, case.seed + 500, n_random)
    t = lambda a: torch.from_numpy(a).to(dev)
    got = (D[t(ls), t(ns), t(ms)] if case.cd_m else D[t(ls), t(ms), t(ns)])
    got = got.double().cpu().numpy()
    D_ref = oracle.gemm_entries(oracle_problem(prep), ms, ns, ls)[0]
    want = oracle.round_to(case.d, D_ref)
    want = want.astype(np.float64) if case.d == "f32" else oracle.decode(case.d, want).reshape(got.shape)
    np.testing.assert_array_equal(got, want)
    assert bool(torch.all(dflat[-GUARD:] == 7.0)), "elements after D were written"
    return gemm.last_config()


def test_output_beyond_2_31_elements(gemm):
    """48000 x 48000 fp16 D (2.3e9 elements, 4.6 GB), row-major."""
    case = Case(M=48000, N=48000, K=16, L=1, ab="f16", c=None, d="f16", alpha=1.5, beta=0.0,
                dist="int2", seed=61)
    cfg = _run_exact(gemm, case)
    assert cfg.tiles * cfg.tile_m * cfg.tile_n >= 48000 * 48000


def test_batch_beyond_2_31_bytes_column_major(gemm):
    """Two batches of 33024 x 33000, D column-major (M contiguous): the second
    batch starts 2.18 GB into D."""
    case = Case(M=33024, N=33000, K=40, L=2, ab="bf16", c=None, d="bf16", cd_m=True,
                alpha=-0.5, beta=0.0, dist="int2", seed=62)
    _run_exact(gemm, case)


def test_long_k_exact(gemm):
    """K = 2^20 (8192 stages of 128 K): integer partial sums stay below 2^22,
    exact in the fp32 accumulator; ragged M and N, fp32 C added."""
    case = Case(M=200, N=264, K=1 << 20, L=1, ab="f16", c="f32", d="f32", alpha=1.0,
                beta=1.0, dist="int2", seed=63)
    cfg = _run_exact(gemm, case, n_random=512)
    assert cfg.tiles < 152             # one wave: each tile runs all 2^20 K

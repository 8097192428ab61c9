"""GPU parity of stream-K: when the tiles fill less than one wave of clusters,
every cluster takes an equal contiguous share of all the tiles' k-blocks and a
tile's owner adds the fp32 partial sums of its earlier k-blocks.  Every case is
compared with the fp64 oracle element by element at the usual bound (the K
summation order changes, not the bound), integer cases bit for bit."""
import pytest
import torch

import dense_gemm_epilogue_persistent_gb300 as G
from gemm_cases import Case, compare_full, prepare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gemm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g = G.Gemm(0)
    yield g
    g.close()


def _force(gemm, cg, bn, epw=0, sk=2, **kw):
    gemm.set_config(cta_group=cg, tile_n=bn, epi_warps=epw, stream_k=sk, **kw)


def _finish(gemm):
    st, detail = gemm.sync_status()
    assert st == G.GEMM_OK, f"device status {G.gemm_status_string(st)} detail={detail:#x}"


def _run_checked(gemm, case, exact=False, expect_sk=True):
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    cfg = gemm.last_config()
    if expect_sk:
        units = cfg.grid_ctas // cfg.cta_group
        assert cfg.stream_k == units and cfg.tiles < units, (cfg.stream_k, cfg.tiles, units)
    compare_full(prep, D, Y, exact=exact)
    return prep, D, Y


# (cta_group, tile_n, epi_warps): single CTAs and pairs, six and ten warps,
# several widths
VARIANTS = [(1, 256, 1), (1, 256, 2), (2, 256, 1), (2, 256, 2), (1, 128, 1), (2, 128, 2),
            (1, 192, 2), (2, 224, 1), (1, 96, 1), (2, 64, 2)]


@pytest.mark.parametrize("variant", VARIANTS)
def test_stream_k_ragged_custom_epilogue(gemm, variant):
    """Ragged M, N and K (K not a multiple of the tile's K, nor the k-blocks a
    multiple of the clusters), f16 C/X/D/Y, batched."""
    cg, bn, epw = variant
    _force(gemm, cg, bn, epw)
    case = Case(M=520, N=392, K=1000, L=2, ab="f16", c="f16", d="f16", x="f16", y="f16",
                alpha=2.0, beta=1.0, xf=3.0, seed=101 + bn)
    _run_checked(gemm, case)
    gemm.set_config(None)


@pytest.mark.parametrize("variant", [(1, 256, 2), (2, 256, 1), (1, 128, 1)])
def test_stream_k_integers_exact(gemm, variant):
    """Integer inputs: every partial and the owner's sum are exact in fp32, so
    D and Y equal the once-rounded oracle bit for bit."""
    cg, bn, epw = variant
    _force(gemm, cg, bn, epw)
    case = Case(M=640, N=512, K=2048, L=1, ab="bf16", c="f32", d="f32", x="f32", y="f32",
                alpha=2.0, beta=-1.0, xf=0.5, dist="int2", seed=7)
    _run_checked(gemm, case, exact=True)
    gemm.set_config(None)


@pytest.mark.parametrize("ab,b,relu", [("bf16", None, False), ("e4m3", None, True),
                                       ("e4m3", "e5m2", False), ("tf32", None, True)])
@pytest.mark.parametrize("layouts", [(False, False, False), (True, True, True)])
def test_stream_k_types_and_layouts(gemm, ab, b, relu, layouts):
    a_mn, b_mn, cd_m = layouts
    if ab == "tf32" and (a_mn or b_mn):
        pytest.skip("tf32 operands are K-major only")
    _force(gemm, 2, 256, 0)
    case = Case(M=1280, N=1024, K=1536, L=1, ab=ab, b=b, c="bf16", d="f16", x="f32", y="bf16",
                a_mn=a_mn, b_mn=b_mn, cd_m=cd_m, alpha=0.75, beta=-0.5, xf=1.25, relu=relu,
                dist="e4m3_pm4" if ab == "e4m3" else "normal1", seed=55)
    _run_checked(gemm, case)
    gemm.set_config(None)


def test_stream_k_single_wave_2048(gemm):
    """The 2048^3 bf16 GEMM with fp32 C/D as 128 x 256 single-CTA tiles and as
    256 x 256 pairs, every element against the oracle."""
    for cg in (1, 2):
        _force(gemm, cg, 256, 2)
        case = Case(M=2048, N=2048, K=2048, L=1, ab="bf16", c="f32", d="f32", alpha=1.0,
                    beta=1.0, dist="uniform1", seed=1)
        _run_checked(gemm, case)
    gemm.set_config(None)


def test_stream_k_deterministic_and_repeated(gemm):
    """The reduction order is fixed: two launches give identical bits; and the
    flags each launch leaves cleared let back-to-back launches on new data
    (no host synchronisation between them) each be right."""
    _force(gemm, 1, 256, 2)
    case = Case(M=1536, N=2048, K=1000, L=1, ab="bf16", c="f32", d="f32", y="f32", alpha=1.0,
                beta=0.5, seed=3)
    prep = prepare(case)
    D1, Y1 = run_gpu(gemm, prep)
    D2, Y2 = run_gpu(gemm, prep)
    _finish(gemm)
    assert torch.equal(D1, D2) and torch.equal(Y1, Y2)
    compare_full(prep, D1, Y1)
    preps = [prepare(Case(M=1536, N=2048, K=1000, L=1, ab="bf16", c="f32", d="f32", y="f32",
                          alpha=1.0, beta=0.5, seed=s)) for s in (11, 12, 13)]
    outs = [run_gpu(gemm, pr) for pr in preps]
    _finish(gemm)
    for pr, (D, Y) in zip(preps, outs):
        compare_full(pr, D, Y)
    gemm.set_config(None)


def test_stream_k_cuda_graph_replay(gemm):
    """Launches captured into a CUDA graph and replayed twice give the same
    results as direct launches (the flags are cleared inside each launch)."""
    _force(gemm, 2, 256, 1)
    case = Case(M=1280, N=1024, K=1536, L=1, ab="bf16", c="f32", d="f32", alpha=1.0, beta=1.0,
                seed=21)
    prep = prepare(case)
    s = torch.cuda.Stream()
    D_ref, _ = run_gpu(gemm, prep)
    _finish(gemm)
    A = prep.A.cuda(); B = prep.B.cuda(); C = prep.C.cuda()
    D = torch.empty_like(D_ref)
    dt = G.make_dtypes("bf16", "f32", "f32")
    launch = lambda: gemm.run(case.M, case.N, case.K, case.L, A, A.shape[-1], 0, B, B.shape[-1],
                              0, C, None, D, None, case.alpha, case.beta, 0.0, dt,
                              s.cuda_stream)
    with torch.cuda.stream(s):
        launch()                                   # plan and encode outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch()
        launch()
    for _ in range(2):
        D.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(D, D_ref)
    _finish(gemm)
    gemm.set_config(None)


def test_stream_k_never_and_not_allowed(gemm):
    """stream_k = 1 turns it off; fp16 accumulators and multi-wave problems do
    not use it even when asked for."""
    case = Case(M=1536, N=2048, K=1000, L=1, ab="bf16", c="f32", d="f32", seed=5)
    _force(gemm, 1, 256, 0, sk=1)
    _run_checked(gemm, case, expect_sk=False)
    assert gemm.last_config().stream_k == 0
    _force(gemm, 2, 256, 0, sk=2)
    case16 = Case(M=1280, N=1024, K=256, L=1, ab="f16", c="f16", d="f16", acc="f16",
                  dist="int2", seed=6)
    _run_checked(gemm, case16, exact=True, expect_sk=False)
    assert gemm.last_config().stream_k == 0
    big = Case(M=4096, N=4096, K=256, L=1, ab="bf16", c="f32", d="f32", seed=8)
    _run_checked(gemm, big, expect_sk=False)
    assert gemm.last_config().stream_k == 0
    gemm.set_config(None)

"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small problems (spanning several tiles and ragged tails) are compared element
by element; the full-size workloads are compared on 4096 seeded entries plus
whole rows and columns at tile boundaries, in the same launch configuration
the benchmark uses.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import dense_gemm_epilogue_persistent_gb300 as G
from gemm_cases import (Case, assert_within, compare_full, compare_sampled, logical,
                        oracle_problem, prepare, run_gpu, to_f64)

pytestmark = pytest.mark.gpu

# (cta_group, tile_n, cluster_m[, cluster_n[, epi_warps]]): single CTAs and CTA
# pairs, 128- and 256-wide tiles, alone and in clusters whose groups share B
# (stacked along M) or A (side by side along N) through TMA multicast, and
# with two epilogue warps per accumulator lane quarter.
VARIANTS = [(1, 128, 1), (1, 256, 1), (2, 128, 1), (2, 256, 1),
            (1, 128, 2), (1, 256, 2), (2, 128, 2), (2, 256, 2),
            (1, 128, 1, 2), (2, 256, 1, 2), (2, 192, 1, 2), (2, 256, 2, 2),
            (1, 128, 1, 1, 2), (2, 256, 1, 1, 2)]
# The other tile widths (multiples of 32 from 64 to 256), alone, in a few
# cluster shapes and with two epilogue warps per lane quarter (odd chunk
# counts: 96 and 224 wide tiles have 3 and 7 chunks).
WIDTH_VARIANTS = [(1, 64, 1), (1, 96, 1), (1, 160, 1), (1, 192, 1), (1, 224, 1),
                  (2, 64, 1), (2, 96, 1), (2, 160, 1), (2, 192, 1), (2, 224, 1),
                  (1, 96, 2), (2, 160, 2), (1, 224, 1, 2), (1, 64, 2, 2),
                  (1, 96, 1, 1, 2), (2, 64, 1, 1, 2), (1, 224, 1, 1, 2), (2, 160, 1, 1, 2)]


def stageable(case, variant):
    """Whether a variant can stage the case's MN-major operands: a CTA's part
    of B (tile_n / cta_group / cluster_m rows) and of A (128 / cluster_n rows)
    must be whole 128-byte atoms."""
    cg, bn, mc = variant[:3]
    nc = variant[3] if len(variant) > 3 else 1
    atom = 128 // W.ELEM_BYTES[case.ab]
    if case.b_mn and (bn // cg // mc) % atom != 0:
        return False
    if case.a_mn and (128 // nc) % atom != 0:
        return False
    return True


@pytest.fixture(scope="module")
def gemm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g = G.Gemm(0)
    yield g
    g.close()


def _force(gemm, cg, bn, mc=1, nc=1, epw=0, stages=0, slots=0):
    gemm.set_config(cta_group=cg, tile_n=bn, cluster_m=mc, cluster_n=nc, epi_warps=epw,
                    stages=stages, epi_slots=slots)


def _finish(gemm):
    st, detail = gemm.sync_status()
    assert st == G.GEMM_OK, f"device status {G.gemm_status_string(st)} detail={detail:#x}"


# ------------------------------------------------------------ bit-exact workload

@pytest.mark.parametrize("variant", VARIANTS + [None])
def test_int256_bit_exact(gemm, variant):
    """256^3, integers in [-2,2], alpha=1.5, beta=-0.5: every intermediate is
    exact in fp32, so D must equal the once-rounded oracle bit for bit."""
    w = W.WORKLOADS["int256_f16_f32"]
    if variant:
        _force(gemm, *variant)
    else:
        gemm.set_config(None)
    prep = prepare(Case.from_workload(w))
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y, exact=True)
    gemm.set_config(None)


@pytest.mark.parametrize("variant", VARIANTS + WIDTH_VARIANTS)
def test_integer_exact_ragged_all_outputs(gemm, variant):
    """Ragged shape, integer inputs, f32 C/X/D/Y: still exact (|acc| < 2^24)."""
    _force(gemm, *variant)
    case = Case(M=300, N=200, K=208, L=2, ab="bf16", c="f32", d="f32", x="f32", y="f32",
                alpha=2.0, beta=-1.0, xf=0.5, dist="int2", seed=7)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y, exact=True)
    gemm.set_config(None)


@pytest.mark.parametrize("variant", VARIANTS)
def test_many_tiles_per_cluster(gemm, variant):
    """Every persistent cluster walks several tiles (4096 x 4096 output), so
    the accumulator double-buffering and the epilogue slot ring wrap around
    many times; all outputs are compared with the oracle."""
    _force(gemm, *variant)
    case = Case(M=4096, N=4096, K=64, L=1, ab="f16", c="f16", d="f16", x="bf16", y="f16",
                alpha=1.0, beta=0.5, xf=-1.0, seed=41)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    cfg = gemm.last_config()
    clusters = cfg.grid_ctas // (cfg.cta_group * cfg.cluster_m * cfg.cluster_n)
    assert cfg.tiles >= 3 * clusters
    compare_full(prep, D, Y)
    gemm.set_config(None)


# ------------------------------------------------------------ reduced-size workloads

SMALL = {
    # custom epilogue, fp16 everywhere
    "efc_f16": Case(M=520, N=392, K=328, L=1, ab="f16", c="f16", d="f16", x="f16", y="f16",
                    alpha=2.0, beta=1.0, xf=3.0, dist="normal1", seed=2),
    # bf16 GEMM with fp32 C/D
    "bf16_f32": Case(M=384, N=640, K=512, L=1, ab="bf16", c="f32", d="f32", alpha=1.0,
                     beta=1.0, dist="uniform1", seed=1),
    # batched, A M-major, B N-major, C/D M-major
    "batched_mn": Case(M=264, N=320, K=200, L=3, ab="bf16", c="bf16", d="bf16", a_mn=True,
                       b_mn=True, cd_m=True, alpha=0.5, beta=0.0, dist="normal002", seed=3),
    # ragged fp8
    "ragged_e4m3": Case(M=300, N=504, K=272, L=1, ab="e4m3", c="f16", d="f16", alpha=0.25,
                        beta=1.0, dist="e4m3_pm4", seed=4),
}


@pytest.mark.parametrize("variant", VARIANTS + WIDTH_VARIANTS + [None])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_workloads(gemm, name, variant):
    case = SMALL[name]
    if variant:
        # MN-major operands are staged (and multicast) in 128-byte atoms
        if not stageable(case, variant):
            pytest.skip("variant cannot stage this MN-major operand")
        _force(gemm, *variant)
    else:
        gemm.set_config(None)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y)
    gemm.set_config(None)


@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("a_mn,b_mn,cd_m", [(False, False, False), (True, False, False),
                                            (False, True, False), (True, True, True),
                                            (False, False, True)])
def test_layouts(gemm, ab, a_mn, b_mn, cd_m):
    case = Case(M=400, N=256, K=320, L=2, ab=ab, c="bf16", d="f32", x="f16", y="bf16",
                a_mn=a_mn, b_mn=b_mn, cd_m=cd_m, alpha=1.5, beta=-0.25, xf=0.75,
                dist="e4m3_pm4" if ab == "e4m3" else "normal1", seed=9)
    gemm.set_config(None)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y)


def test_layout_equivalence_bitwise(gemm):
    """The same logical values in every layout give identical outputs."""
    base = None
    for a_mn in (False, True):
        for b_mn in (False, True):
            for cd_m in (False, True):
                case = Case(M=256, N=256, K=192, L=2, ab="f16", c="f16", d="f16", y="f32",
                            a_mn=a_mn, b_mn=b_mn, cd_m=cd_m, alpha=1.25, beta=0.5, seed=12)
                gemm.set_config(None)
                prep = prepare(case)
                D, Y = run_gpu(gemm, prep)
                _finish(gemm)
                out = (logical(D, cd_m), logical(Y, cd_m))
                if base is None:
                    base = out
                else:
                    assert torch.equal(base[0], out[0]) and torch.equal(base[1], out[1])


# ------------------------------------------------------------ shared operands

@pytest.mark.parametrize("variant", [(2, 256, 1, 2), (1, 128, 1, 2), (2, 256, 2, 2),
                                     (2, 128, 2, 1), (1, 192, 2, 2)])
@pytest.mark.parametrize("ab", ["bf16", "e4m3"])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, False), (False, True),
                                       (True, True)])
def test_shared_operand_layouts(gemm, variant, ab, a_mn, b_mn):
    """Clusters that share A (along N) and/or B (along M) by multicast, with
    K-major and MN-major operands, on a ragged shape whose last cluster tiles
    have groups entirely outside the output (rows 768.. and columns 768.. of a
    720 x 704 output)."""
    case = Case(M=720, N=704, K=400, L=2, ab=ab, c="f16", d="f32", x="bf16", y="f16",
                a_mn=a_mn, b_mn=b_mn, alpha=-0.75, beta=1.0, xf=0.5,
                dist="e4m3_pm4" if ab == "e4m3" else "normal1", seed=31)
    if not stageable(case, variant):
        pytest.skip("variant cannot stage this MN-major operand")
    _force(gemm, *variant)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    cfg = gemm.last_config()
    assert (cfg.cluster_m, cfg.cluster_n) == (variant[2], variant[3])
    compare_full(prep, D, Y)
    gemm.set_config(None)


# ------------------------------------------------------- two epilogue warps per lane quarter

@pytest.mark.parametrize("cg,bn", [(1, 128), (2, 256), (1, 224)])
@pytest.mark.parametrize("slots", [2, 3, 4, 6])
@pytest.mark.parametrize("loads", [True, False])
def test_two_epilogue_warps_per_quarter(gemm, cg, bn, slots, loads):
    """Eight epilogue warps, the two of each lane quarter taking alternate
    32-column chunks with half the slots each (one slot each at 2 and 3
    slots: loads wait for the previous store), over many tiles per CTA; with
    and without C/X loads.  All outputs against the oracle."""
    case = Case(M=4608, N=2080, K=96, L=1, ab="bf16", c="f16" if loads else None, d="f16",
                x="bf16" if loads else None, y="f16", alpha=1.5, beta=-0.5 if loads else 0.0,
                xf=2.0 if loads else 0.0, seed=slots * 7 + bn + cg)
    _force(gemm, cg, bn, 1, 1, 2, 2 if slots > 2 else 0, slots)   # short ring: room for slots
    prep = prepare(case)
    try:
        D, Y = run_gpu(gemm, prep)
    except G.GemmError:
        gemm.set_config(None)
        pytest.skip("that many slots do not fit beside the ring")
    _finish(gemm)
    cfg = gemm.last_config()
    assert (cfg.epi_warps, cfg.epi_slots, cfg.tile_n) == (2, slots, bn)
    clusters = cfg.grid_ctas // cfg.cta_group
    assert cfg.tiles >= 2 * clusters
    compare_full(prep, D, Y)
    gemm.set_config(None)


@pytest.mark.parametrize("epi", [
    dict(c="f16", x="bf16", y="f16", d="f16", beta=-0.75, xf=1.5, relu=False),
    dict(c="f16", x="bf16", y=None, d="bf16", beta=0.5, xf=-2.0, relu=True),
    dict(c="f32", x=None, y="f32", d="f32", beta=1.0, xf=0.0, relu=False),
    dict(c="bf16", x=None, y=None, d="f16", beta=0.25, xf=0.0, relu=True),
    dict(c=None, x="f16", y="bf16", d="f32", beta=0.0, xf=0.5, relu=False),
    dict(c=None, x=None, y=None, d="bf16", beta=0.0, xf=0.0, relu=False),
])
@pytest.mark.parametrize("cd_m", [False, True])
@pytest.mark.parametrize("ab,acc", [("bf16", "f32"), ("e4m3", "f16"), ("tf32", "f32")])
def test_epilogue_warp_forms_bitwise_equal(gemm, epi, cd_m, ab, acc):
    """The ten-warp form folds C and X into D piece by piece after the
    accumulator load; the six-warp form reads whole rows first.  Both apply the
    same operations in the same order, so on the same tile their D and Y are
    bit-identical (real-valued inputs, every epilogue shape)."""
    case = Case(M=640, N=544, K=264 if ab != "e4m3" else 256, L=2, ab=ab, c=epi["c"],
                d=epi["d"], x=epi["x"], y=epi["y"], cd_m=cd_m, alpha=0.875, beta=epi["beta"],
                xf=epi["xf"], relu=epi["relu"], acc=acc,
                dist="e4m3_pm4" if ab == "e4m3" else "normal1", seed=77 + cd_m)
    prep = prepare(case)
    outs = []
    for epw in (1, 2):
        _force(gemm, 2, 224, 1, 1, epw)
        D, Y = run_gpu(gemm, prep)
        _finish(gemm)
        assert gemm.last_config().epi_warps == epw
        outs.append((D.clone(), None if Y is None else Y.clone()))
    gemm.set_config(None)
    assert torch.equal(outs[0][0].view(torch.uint8), outs[1][0].view(torch.uint8))
    if outs[0][1] is not None:
        assert torch.equal(outs[0][1].view(torch.uint8), outs[1][1].view(torch.uint8))
    compare_full(prep, *outs[1])


def test_two_epilogue_warps_need_one_group_clusters(gemm):
    """Two epilogue warps per quarter exist only for clusters of one CTA group."""
    case = SMALL["efc_f16"]
    prep = prepare(case)
    gemm.set_config(cta_group=2, tile_n=256, cluster_m=2, epi_warps=2)
    with pytest.raises(G.GemmError):
        run_gpu(gemm, prep)
    gemm.set_config(None)


# ------------------------------------------------------------ split last wave

@pytest.mark.parametrize("variant,shape", [
    ((2, 192, 1), (2560, 1920, 192)),      # 100 tiles on 76 pairs: 24 split
    ((1, 64, 1), (1280, 2048, 128)),       # 320 tiles on 152 CTAs: 16 split
    ((2, 256, 1), (2560, 2560, 192)),      # 100 tiles on 76 pairs: 24 split
    ((1, 256, 1), (2048, 2560, 128)),      # 160 tiles on 152 CTAs: 8 split
    ((1, 128, 1), (2048, 1280, 256)),
    ((2, 128, 1), (2048, 1408, 128)),
    ((2, 256, 1), (2500, 2552, 200)),      # ragged
    ((1, 256, 1), (2000, 2560, 136)),
    ((1, 64, 1, 1, 2), (1280, 2048, 128)),    # half items of one chunk: one warp idle
    ((2, 192, 1, 1, 2), (2560, 1920, 192)),   # half items of three chunks
    ((2, 256, 1, 1, 2), (2500, 2552, 200)),
])
def test_split_last_wave(gemm, variant, shape):
    """Tiles of the last, partial wave run as two half-width items each."""
    M, N, K = shape
    _force(gemm, *variant)
    case = Case(M=M, N=N, K=K, L=1, ab="f16", c="f16", d="f16", x="bf16", y="f16", alpha=1.0,
                beta=-0.5, xf=2.0, seed=M + N)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    cfg = gemm.last_config()
    assert cfg.tail_split > 0
    compare_full(prep, D, Y)
    gemm.set_config(None)


@pytest.mark.parametrize("ab,b_mn", [("bf16", True), ("e4m3", False), ("tf32", False)])
def test_split_last_wave_types_and_layouts(gemm, ab, b_mn):
    _force(gemm, 2 if ab == "bf16" else 1, 256, 1)
    case = Case(M=2048, N=2560, K=256, L=1, ab=ab, c="f32", d="f32", y="bf16", b_mn=b_mn,
                alpha=0.5, beta=1.0, dist="e4m3_pm4" if ab == "e4m3" else "normal1", seed=71)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    assert gemm.last_config().tail_split > 0
    compare_full(prep, D, Y)
    gemm.set_config(None)


# ------------------------------------------------------------ fp8 pairs, relu epilogue

@pytest.mark.parametrize("variant", [None, (1, 256, 1), (2, 256, 1), (2, 256, 2), (1, 128, 1)])
@pytest.mark.parametrize("a_dt,b_dt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("relu", [False, True])
def test_fp8_pairs_and_relu(gemm, variant, a_dt, b_dt, relu):
    """E5M2 inputs, mixed E4M3 x E5M2 pairs (tcgen05 kind::f8f6f4 with two
    operand formats) and the relu epilogue, on ragged shapes."""
    if variant:
        _force(gemm, *variant)
    else:
        gemm.set_config(None)
    case = Case(M=700, N=520, K=400, L=2, ab=a_dt, b=None if b_dt == a_dt else b_dt, c="f16",
                d="f16", x="bf16", y="f32", alpha=0.25, beta=1.0, xf=0.5, relu=relu,
                dist="e4m3_pm4", seed=61)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y)
    gemm.set_config(None)


@pytest.mark.parametrize("layouts", [(True, True, True), (False, True, False)])
def test_fp8_pair_mn_major(gemm, layouts):
    a_mn, b_mn, cd_m = layouts
    case = Case(M=512, N=512, K=256, L=1, ab="e5m2", b="e4m3", c="f32", d="bf16", a_mn=a_mn,
                b_mn=b_mn, cd_m=cd_m, alpha=1.0, beta=-0.5, relu=True, dist="e4m3_pm4", seed=63)
    gemm.set_config(None)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y)


# ------------------------------------------------------------ tf32 inputs

@pytest.mark.parametrize("variant", [None, (1, 256, 1), (2, 256, 1), (2, 256, 2), (1, 128, 1),
                                     (2, 128, 1)])
def test_tf32(gemm, variant):
    """tf32 operands (fp32 storage of tf32 values, K-major, tcgen05 kind::tf32)."""
    if variant:
        _force(gemm, *variant)
    else:
        gemm.set_config(None)
    case = Case(M=600, N=456, K=200, L=2, ab="tf32", c="f32", d="f32", x="f16", y="bf16",
                alpha=1.5, beta=-1.0, xf=0.25, dist="normal1", seed=65)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y)
    gemm.set_config(None)


def test_tf32_integers_exact(gemm):
    case = Case(M=256, N=384, K=512, L=1, ab="tf32", c="f32", d="f32", y="f32", alpha=1.0,
                beta=1.0, dist="int2", seed=67)
    gemm.set_config(None)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y, exact=True)


def test_tf32_general_fp32_inputs(gemm):
    """GEMM_TF32 on fp32 values that are NOT tf32 values (low 13 fraction bits
    set).  The tensor core reads sign, exponent and the upper 10 fraction bits
    (truncated or rounded: either way each operand is off by less than 2^-10
    relative), so each product is off by less than 2^-9 + 2^-20 relative and
    the accumulator bound gains that term: |D - ref| <= (2^-9 + 2^-20 + 2^-10)
    |alpha| sum|ab| + 2^-10 (|beta c| + |x_factor x|) against the exact result
    on the fp32 values as given."""
    case = Case(M=384, N=520, K=264, L=1, ab="tf32", c="f32", d="f32", x="f32", y="f32",
                alpha=1.25, beta=0.5, xf=-2.0, dist="normal1", seed=68)
    prep = prepare(case)
    g = torch.Generator().manual_seed(1068)
    prep.A = torch.randn(case.L, case.M, case.K, generator=g).contiguous()
    prep.B = torch.randn(case.L, case.N, case.K, generator=g).contiguous()
    low = lambda t: (t.view(torch.int32) & 0x1FFF) != 0
    assert low(prep.A).float().mean() > 0.99 and low(prep.B).float().mean() > 0.99
    gemm.set_config(None)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    D_ref, Y_ref, S = oracle.gemm(oracle_problem(prep))
    Cv, Xv = to_f64(prep.inp.C), to_f64(prep.inp.X)
    acc_bound = (2.0 ** -9 + 2.0 ** -20 + 2.0 ** -10) * S
    assert_within("D", to_f64(D), D_ref,
                  abs(case.alpha) * acc_bound + 2.0 ** -10 * (abs(case.beta * Cv) +
                                                              abs(case.xf * Xv)))
    assert_within("Y", to_f64(Y), Y_ref, acc_bound)
    # the operands' low bits are really dropped: Y is farther from the exact
    # product of the fp32 values than fp32 accumulation of exact tf32 operands
    # puts it (about 2^-20 of sum|ab| at this K)
    assert np.max(np.abs(to_f64(Y) - Y_ref) / S) > 2.0 ** -17


# ------------------------------------------------------------ fp16 accumulator

def _int_fp8_inputs(case):
    """Integer inputs in [-2, 2] stored as fp8 codes (exact in E4M3 and E5M2),
    with integer C: every running sum stays an integer below 2048."""
    g = torch.Generator().manual_seed(case.seed)
    fp8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
    A = torch.randint(-2, 3, (case.L, case.M, case.K), generator=g).float()
    B = torch.randint(-2, 3, (case.L, case.N, case.K), generator=g).float()
    C = torch.randint(-2, 3, (case.L, case.M, case.N), generator=g).float()
    return W.Inputs(A.to(fp8[case.ab]).view(torch.uint8),
                    B.to(fp8[case.b or case.ab]).view(torch.uint8), C, None)


@pytest.mark.parametrize("variant", VARIANTS + [None])
@pytest.mark.parametrize("ab", ["f16", "e4m3"])
def test_f16_accumulator_integers_exact(gemm, variant, ab):
    """fp16 accumulation, integer inputs in [-2, 2], K = 400: every running
    sum is an integer of magnitude <= 1600 < 2048, exact in fp16 whatever the
    rounding points, so Y and D (f32, alpha 1.5, beta -0.5) are bit-exact."""
    if variant:
        _force(gemm, *variant)
    else:
        gemm.set_config(None)
    case = Case(M=300, N=264, K=400, L=2, ab=ab, c="f32", d="f32", y="f32", alpha=1.5,
                beta=-0.5, dist="int2", seed=71, acc="f16")
    prep = prepare(case, _int_fp8_inputs(case) if ab != "f16" else None)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y, exact=True)
    gemm.set_config(None)


@pytest.mark.parametrize("variant", [None, (1, 128, 1), (1, 256, 2), (2, 128, 1), (2, 256, 1)])
@pytest.mark.parametrize("ab,b", [("f16", None), ("e4m3", None), ("e5m2", "e4m3")])
def test_f16_accumulator_bound_and_precision(gemm, variant, ab, b):
    """fp16 accumulation on real-valued ragged problems: D and Y within the
    fp16-accumulator bound, and Y (stored as f32) holds fp16 values only --
    the accumulator really is fp16 (an fp32 accumulator would not round
    there).  The same problem with an fp32 accumulator is closer to the
    exact result on average."""
    if variant:
        _force(gemm, *variant)
    else:
        gemm.set_config(None)
    dist = "normal1" if ab == "f16" else "e4m3_pm4"
    case = Case(M=520, N=392, K=1008, L=2, ab=ab, b=b, c="f16", d="f16", x="bf16", y="f32",
                alpha=0.75, beta=1.0, xf=-0.5, dist=dist, seed=73, acc="f16")
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    _, Y_ref = compare_full(prep, D, Y)
    y = Y.cpu()
    assert torch.equal(y, y.half().float())
    prep32 = prepare(Case(**{**case.__dict__, "acc": "f32"}), prep.inp)
    _, Y32 = run_gpu(gemm, prep32)
    _finish(gemm)
    err16 = np.abs(to_f64(logical(Y, False)) - Y_ref).mean()
    err32 = np.abs(to_f64(logical(Y32, False)) - Y_ref).mean()
    assert err32 < err16
    gemm.set_config(None)


def test_f16_accumulator_overflows_to_infinity(gemm):
    """The fp16 accumulator's documented range: all-16 inputs give running sums
    of 256 per k; at K = 240 the result (61440) is exact, from K = 256 on the
    sum passes the fp16 maximum (65504) and Y and D are infinite (no
    saturation)."""
    gemm.set_config(None)
    dev = torch.device("cuda")
    dt = G.make_dtypes("f16", "f32", "f32", "f32", "f32", acc="f16")
    for K, want in ((240, 61440.0), (256, float("inf")), (512, float("inf"))):
        A = torch.full((1, 128, K), 16.0, dtype=torch.float16, device=dev)
        B = torch.full((1, 136, K), 16.0, dtype=torch.float16, device=dev)
        D = torch.empty(1, 128, 136, dtype=torch.float32, device=dev)
        Y = torch.empty(1, 128, 136, dtype=torch.float32, device=dev)
        gemm.run(128, 136, K, 1, A, K, 0, B, K, 0, None, None, D, Y, 0.5, 0.0, 0.0, dt)
        _finish(gemm)
        assert torch.all(Y == want) and torch.all(D == 0.5 * want), K


def test_f16_accumulator_split_last_wave(gemm):
    """fp16 accumulation through the half-width items of a split last wave
    (100 pair tiles on 76 pairs: 24 split; the half-width instruction
    descriptor carries the fp16 accumulator format too)."""
    _force(gemm, 2, 256, 1)
    case = Case(M=2560, N=2560, K=192, L=1, ab="f16", c="f16", d="f16", y="f16", alpha=1.0,
                beta=1.0, dist="normal1", seed=75, acc="f16")
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    assert gemm.last_config().tail_split > 0
    compare_full(prep, D, Y)
    gemm.set_config(None)


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("M,N,K,L", [(8, 8, 16, 1), (1, 8, 16, 1), (129, 136, 72, 1),
                                     (130, 264, 1000, 3), (2048, 8, 64, 1), (8, 2000, 16, 2)])
def test_ragged_shapes(gemm, M, N, K, L):
    case = Case(M=M, N=N, K=K, L=L, ab="f16", c="f16", d="f16", y="f16", alpha=1.0, beta=2.0,
                seed=M + N + K)
    gemm.set_config(None)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y)


@pytest.mark.parametrize("M,N,K,L,cd_m,variant", [
    (64, 64, 32, 257, False, None), (40, 72, 48, 300, False, (2, 128, 1)),
    (1, 8, 64, 129, False, None), (136, 1, 16, 65, True, (1, 128, 2)),
])
def test_many_small_batches(gemm, M, N, K, L, cd_m, variant):
    """Batched problems with many small, ragged members: batch index, tile
    order across batches and the last-wave split all in play.  (A single
    column needs column-major C/D: the packed leading dimension must be
    16-byte aligned.)"""
    if variant:
        _force(gemm, *variant)
    else:
        gemm.set_config(None)
    case = Case(M=M, N=N, K=K, L=L, ab="bf16", c="f32", d="f16", y="f32", cd_m=cd_m,
                alpha=0.5, beta=-1.0, seed=M * 7 + L)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, Y)
    gemm.set_config(None)


def test_k_zero(gemm):
    case = Case(M=200, N=136, K=0, L=2, ab="bf16", c="f32", d="f32", x="f16", y="f32",
                alpha=3.0, beta=0.5, xf=-2.0, seed=5)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    D_ref, Y_ref = compare_full(prep, D, Y, exact=True)
    assert np.all(Y_ref == 0)


def test_empty_problems_are_noops(gemm):
    D = torch.full((4, 16), 7.0, device="cuda")
    dt = G.make_dtypes("f16")
    for M, N, L in [(0, 16, 1), (4, 0, 1), (4, 16, 0)]:
        st = G.gemm_run(gemm.handle, M, N, 32, L, 0, 32, 0, 0, 32, 0, 0, 0, D, 0, 1.0, 0.0, 0.0,
                        dt)
        assert st == G.GEMM_OK
    _finish(gemm)
    assert torch.all(D == 7.0)


def test_inputs_unchanged_canaries_and_alias(gemm):
    """C and X are read-only, nothing outside D and Y is written, and D may
    alias C (each element of C is read before it is overwritten)."""
    case = Case(M=200, N=264, K=136, L=2, ab="f16", c="f16", d="f16", x="f16", y="f16",
                alpha=1.0, beta=1.0, xf=2.0, seed=17)
    prep = prepare(case)
    dev = torch.device("cuda")
    n = case.L * case.M * case.N
    pad = 4096
    Dbuf = torch.full((n + 2 * pad,), 1234.0, dtype=torch.float16, device=dev)
    Ybuf = torch.full((n + 2 * pad,), -77.0, dtype=torch.float16, device=dev)
    D = Dbuf[pad:pad + n].view(case.L, case.M, case.N)
    Y = Ybuf[pad:pad + n].view(case.L, case.M, case.N)
    C_dev = prep.C.to(dev)
    X_dev = prep.X.to(dev)
    D, Y = run_gpu(gemm, prep, D=D, Y=Y, C_dev=C_dev, X_dev=X_dev)
    _finish(gemm)
    assert torch.equal(C_dev.cpu(), prep.C) and torch.equal(X_dev.cpu(), prep.X)
    for buf, v in ((Dbuf, 1234.0), (Ybuf, -77.0)):
        assert torch.all(buf[:pad] == v) and torch.all(buf[pad + n:] == v)
    compare_full(prep, D, Y)
    # alias: D == C
    C_alias = prep.C.to(dev)
    D2, _ = run_gpu(gemm, prep, D=C_alias, C_dev=C_alias)
    _finish(gemm)
    assert torch.equal(D2.cpu(), D.cpu())


def test_beta_zero_does_not_read_C(gemm):
    case = Case(M=136, N=128, K=64, L=1, ab="bf16", c="f32", d="f32", alpha=1.0, beta=0.0,
                seed=23)
    prep = prepare(case)
    C_nan = torch.full_like(prep.C, float("nan")).cuda()
    D, _ = run_gpu(gemm, prep, C_dev=C_nan)
    _finish(gemm)
    assert not torch.isnan(D).any()
    compare_full(prep, D, None)


def test_x_null_means_no_x_term(gemm):
    case = Case(M=256, N=256, K=128, L=1, ab="f16", c="f16", d="f16", x="f16", y="f16",
                alpha=1.0, beta=1.0, xf=3.0, seed=29)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep, use_x=False)
    _finish(gemm)
    compare_full(prep, D, Y, use_x=False)


def test_lda_ldb_padding(gemm):
    case = Case(M=200, N=136, K=100, L=2, ab="bf16", c="f32", d="f32", alpha=1.0, beta=0.5,
                lda_pad=28, ldb_pad=12, seed=31)
    prep = prepare(case)
    D, _ = run_gpu(gemm, prep)
    _finish(gemm)
    compare_full(prep, D, None)


def test_dependent_launch_chain(gemm):
    """Back-to-back dependent GEMMs on one stream, no host syncs (the kernel is
    launched with programmatic stream serialization and waits on the previous
    grid before touching global memory): D1 = A1 B1^T feeds GEMM 2 as A
    (read after write), and GEMM 3 overwrites GEMM 2's B (write after read).
    Integer inputs keep every value exact, so each iteration's D2 must equal
    the oracle bit for bit."""
    gemm.set_config(None)
    g = torch.Generator().manual_seed(91)
    M, K, N, N2 = 256, 64, 128, 192
    ri = lambda *sh: torch.randint(-2, 3, sh, generator=g).to(torch.float16)
    A1, B1, B2 = ri(1, M, K), ri(1, N, K), ri(1, N2, N)
    dev = torch.device("cuda")
    A1d, B1d, B2_orig = A1.to(dev), B1.to(dev), B2.to(dev)
    B2d = torch.empty_like(B2_orig)
    D1 = torch.empty(1, M, N, dtype=torch.float16, device=dev)
    A3 = torch.ones(1, N2, K, dtype=torch.float16, device=dev)
    dt16 = G.make_dtypes("f16", "f32", "f16")
    dt32 = G.make_dtypes("f16", "f32", "f32")
    outs = []
    for it in range(12):
        B2d.copy_(B2_orig)
        gemm.run(M, N, K, 1, A1d, K, 0, B1d, K, 0, None, None, D1, None, 1.0, 0.0, 0.0, dt16)
        D2 = torch.empty(1, M, N2, dtype=torch.float32, device=dev)
        gemm.run(M, N2, N, 1, D1, N, 0, B2d, N, 0, None, None, D2, None, 1.0, 0.0, 0.0, dt32)
        # overwrite GEMM 2's B with (A3 B1^T), a different integer matrix
        gemm.run(N2, N, K, 1, A3, K, 0, B1d, K, 0, None, None, B2d, None, 1.0, 0.0, 0.0, dt16)
        outs.append(D2)
    _finish(gemm)
    st = W.storage_view_np
    p1 = oracle.Problem(M, N, K, 1, st(A1), K, False, st(B1), K, False, None, None, "f16", alpha=1.0)
    D1_ref = oracle.round_to("f16", oracle.gemm(p1)[0])        # exact integers in fp16 storage
    p2 = oracle.Problem(M, N2, N, 1, D1_ref, N, False, st(B2), N, False, None, None, "f16",
                        alpha=1.0)
    want = oracle.gemm(p2)[0].astype(np.float32)
    for D2 in outs:
        np.testing.assert_array_equal(D2.cpu().numpy(), want)


def test_cuda_graph_capture_and_replay(gemm):
    """gemm_run calls captured into a CUDA graph (a dependent chain: D1 feeds
    the second GEMM) replay to the same bits as the eager calls, also after
    the inputs behind the captured pointers change."""
    gemm.set_config(None)
    g = torch.Generator().manual_seed(93)
    M, K, N, N2 = 384, 128, 256, 192
    dev = torch.device("cuda")
    A1 = torch.randn(1, M, K, generator=g).to(torch.float16).to(dev)
    B1 = torch.randn(1, N, K, generator=g).to(torch.float16).to(dev)
    B2 = torch.randn(1, N2, N, generator=g).to(torch.float16).to(dev)
    C2 = torch.randn(1, M, N2, generator=g).to(dev)
    D1 = torch.empty(1, M, N, dtype=torch.float16, device=dev)
    D2 = torch.empty(1, M, N2, dtype=torch.float32, device=dev)
    dt16 = G.make_dtypes("f16", "f32", "f16")
    dt32 = G.make_dtypes("f16", "f32", "f32")
    s = torch.cuda.Stream()

    def chain():
        gemm.run(M, N, K, 1, A1, K, 0, B1, K, 0, None, None, D1, None, 1.0, 0.0, 0.0, dt16, s)
        gemm.run(M, N2, N, 1, D1, N, 0, B2, N, 0, C2, None, D2, None, 0.5, -1.0, 0.0, dt32, s)

    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    want1, want2 = D1.clone(), D2.clone()
    graph = torch.cuda.CUDAGraph()
    D1.zero_(); D2.zero_()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        chain()
    for _ in range(3):
        D1.zero_(); D2.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(D1, want1) and torch.equal(D2, want2)
    # new data behind the captured pointers: the replay reads it
    A1.mul_(-1)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(D1, -want1)
    st, detail = gemm.sync_status()
    assert st == G.GEMM_OK, detail


def test_launch_cache_reuse_and_eviction(gemm):
    """The handle caches prepared launches (plan, tensor maps, parameters) per
    distinct call.  Six distinct problems cycled three times evict and refill
    the cache; every result stays bit-exact, a forced configuration between
    two identical calls takes effect, and new data behind the same pointers is
    read anew."""
    gemm.set_config(None)
    shapes = [(256, 256, 64), (384, 128, 128), (128, 512, 64), (512, 256, 32), (256, 384, 96),
              (640, 128, 64)]
    cases = [Case(M=m, N=n, K=k, L=1, ab="f16", c="f32", d="f32", alpha=1.5, beta=-0.5,
                  dist="int2", seed=100 + i) for i, (m, n, k) in enumerate(shapes)]
    preps = [prepare(c) for c in cases]
    for rnd in range(3):
        for prep in preps:
            D, Y = run_gpu(gemm, prep)
            _finish(gemm)
            compare_full(prep, D, Y, exact=True)
    # identical call, forced configuration in between
    prep = preps[0]
    dev = torch.device("cuda")
    A, B, C = prep.A.to(dev), prep.B.to(dev), prep.C.to(dev)
    D = torch.empty(1, 256, 256, dtype=torch.float32, device=dev)
    dt = G.make_dtypes("f16", "f32", "f32")
    args = (256, 256, 64, 1, A, 64, 0, B, 64, 0, C, None, D, None, 1.5, -0.5, 0.0, dt)
    gemm.run(*args)
    first = gemm.last_config()
    alt = (1, 128) if (first.cta_group, first.tile_n) != (1, 128) else (2, 256)
    gemm.set_config(cta_group=alt[0], tile_n=alt[1])
    gemm.run(*args)
    forced = gemm.last_config()
    assert (forced.cta_group, forced.tile_n) == alt
    _finish(gemm)
    compare_full(prep, D, None, exact=True)
    # same pointers, new contents
    A.zero_()
    gemm.run(*args)
    _finish(gemm)
    want = oracle.round_to("f32", -0.5 * to_f64(prep.inp.C))
    np.testing.assert_array_equal(D.cpu().numpy(), want)
    gemm.set_config(None)


def _run_host(gemm, prep, pinned=True, stream=None):
    """gemm_run_host on the CPU storage of a prepared case.  Returns the host D
    and Y (valid once the stream has passed the call) and the host inputs,
    which the caller keeps alive until then (the copies read them
    asynchronously)."""
    from gemm_cases import out_shape
    c = prep.case
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    A, B = pin(prep.A), pin(prep.B)
    C = pin(prep.C) if prep.C is not None else None
    X = pin(prep.X) if prep.X is not None else None
    D = torch.empty(out_shape(c), dtype=W.TORCH_DTYPE[c.d], pin_memory=pinned)
    Y = torch.empty(out_shape(c), dtype=W.TORCH_DTYPE[c.y], pin_memory=pinned) if c.y else None
    dt = G.make_dtypes(c.ab, c.c or "f32", c.d, c.x or "f32", c.y or "f32",
                       G.GEMM_MN_MAJOR if c.cd_m else G.GEMM_K_MAJOR, b=c.b,
                       epilogue=G.GEMM_EPI_RELU if c.relu else G.GEMM_EPI_LINEAR, acc=c.acc)
    gemm.run_host(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B, B.shape[-1], int(c.b_mn),
                  C, X, D, Y, c.alpha, c.beta, c.xf, dt, stream)
    return D, Y, (A, B, C, X)


def test_run_host_matches_device_path(gemm):
    """gemm_run_host (host buffers, copies through the handle's workspace) gives
    the device path's bits: pinned and pageable buffers, an M-major A with a
    padded leading dimension, batches, C/X/D/Y, a workspace that grows then is
    reused by a smaller call, and K = 0."""
    gemm.set_config(None)
    cases = [
        Case(M=296, N=264, K=200, L=2, ab="f16", c="f16", d="f16", x="bf16", y="f32",
             a_mn=True, lda_pad=8, alpha=1.5, beta=-0.5, xf=0.25, seed=95),
        Case(M=1024, N=1536, K=512, L=1, ab="bf16", c="f32", d="bf16", y="bf16", b_mn=True,
             cd_m=True, alpha=1.0, beta=1.0, seed=96),
        Case(M=200, N=136, K=0, L=3, ab="f16", c="f32", d="f32", x="f16", alpha=1.0, beta=2.0,
             xf=-1.0, seed=97),
        Case(M=384, N=512, K=256, L=1, ab="e4m3", b="e5m2", c="f16", d="f16", relu=True,
             alpha=0.5, beta=1.0, dist="e4m3_pm4", seed=98),
    ]
    for pinned in (True, False):
        for case in cases:
            prep = prepare(case)
            D_dev, Y_dev = run_gpu(gemm, prep)
            D, Y, keep = _run_host(gemm, prep, pinned)
            _finish(gemm)
            del keep
            assert torch.equal(D, D_dev.cpu()), (case, pinned)
            if Y is not None:
                assert torch.equal(Y, Y_dev.cpu()), (case, pinned)


def test_run_host_two_handles_overlap(gemm):
    """Calls on host buffers overlap across two handles on two streams (each
    handle owns its workspace); every result matches the device path."""
    gemm.set_config(None)
    h2 = G.Gemm(0)
    try:
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        handles = [gemm, h2]
        preps = [prepare(Case(M=512, N=640, K=384, L=2, ab="f16", c="f16", d="f16", y="f16",
                              alpha=1.0, beta=0.5, seed=110 + i)) for i in range(6)]
        want = [tuple(t.cpu() for t in run_gpu(gemm, pr)) for pr in preps]
        _finish(gemm)
        got = []
        for i, pr in enumerate(preps):
            got.append(_run_host(handles[i % 2], pr, True, streams[i % 2].cuda_stream))
        torch.cuda.synchronize()
        for (D, Y, _), (Dw, Yw) in zip(got, want):
            assert torch.equal(D, Dw) and torch.equal(Y, Yw)
        st, _ = h2.sync_status()
        assert st == G.GEMM_OK
    finally:
        h2.close()


def test_streams_and_repeat_determinism(gemm):
    case = SMALL["efc_f16"]
    prep = prepare(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        D1, Y1 = run_gpu(gemm, prep, stream=s)
        D2, Y2 = run_gpu(gemm, prep, stream=s)
    st, _ = gemm.sync_status(s)
    assert st == G.GEMM_OK
    assert torch.equal(D1, D2) and torch.equal(Y1, Y2)


# ------------------------------------------------------------ full-size workloads

FULL = ["gemm2048_bf16_f32", "efc8192_f16", "gemm8192_bf16", "batched16_bf16_mn",
        "ragged_e4m3_f16", "e5m2_4096_f16", "fp8mix_relu_4096", "tf32_4096_f32",
        "f16acc_4096_f16", "e4m3_f16acc_4096"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_sampled(gemm, name):
    """Each full-size workload in the launch configuration the benchmark uses
    (automatic selection), checked on sampled entries and boundary lines."""
    w = W.WORKLOADS[name]
    gemm.set_config(None)
    case = Case.from_workload(w)
    prep = prepare(case)
    D, Y = run_gpu(gemm, prep)
    _finish(gemm)
    cfg = gemm.last_config()
    n = compare_sampled(prep, D, Y, cfg.tile_m, cfg.tile_n, seed=w.seed + 1000)
    assert n >= 4096

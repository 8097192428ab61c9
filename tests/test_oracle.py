"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties the oracle to what the pages or the mathematics fix:
library decoders and rounding, exact rational brute force, closed forms,
special cases that reduce to a library matmul, and invariants of the
definition Y = A*B, D = alpha*A*B + beta*C + x_factor*X with B stored N x K
("custom_epilogue_dense_gemm.py", module docstring; "04_mma_tma_2sm_sm100.cu",
header comment).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- helpers

def _storage(t):
    return W.storage_view_np(t)


def _problem(A, B, C=None, X=None, *, ab="f16", c="f32", x="f32", a_mn=False, b_mn=False,
             cd_m=False, alpha=1.0, beta=0.0, xf=0.0, use_c=None, use_x=None, lda=None, ldb=None,
             b=None, relu=False, acc_chunk=0):
    """Build an oracle Problem from LOGICAL torch tensors A [L,M,K], B [L,N,K],
    C/X [L,M,N] (storage dtypes), laying them out as requested."""
    L, M, K = A.shape
    N = B.shape[1]
    As = W.to_storage(A, a_mn)
    Bs = W.to_storage(B, b_mn)
    if lda is not None:          # pad the leading dimension with junk
        pad = lda - As.shape[2]
        As = torch.cat([As, torch.full((L, As.shape[1], pad), 7, dtype=As.dtype)], 2).contiguous()
    if ldb is not None:
        pad = ldb - Bs.shape[2]
        Bs = torch.cat([Bs, torch.full((L, Bs.shape[1], pad), 7, dtype=Bs.dtype)], 2).contiguous()
    Cs = None if C is None else _storage(W.to_storage(C, cd_m))
    Xs = None if X is None else _storage(W.to_storage(X, cd_m))
    return oracle.Problem(M, N, K, L, _storage(As), As.shape[2], a_mn, _storage(Bs), Bs.shape[2],
                          b_mn, Cs, Xs, ab, c, x, cd_m, alpha, beta, xf, use_c, use_x, b, relu,
                          acc_chunk)


def _f64(t, fp8="e4m3"):
    if t.dtype == torch.uint8:   # fp8 codes
        return t.view(torch.float8_e4m3fn if fp8 == "e4m3" else torch.float8_e5m2).double()
    return t.double()


# ---------------------------------------------------------------- decoders

def test_decode_f16_matches_numpy_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = oracle.decode("f16", codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_decode_bf16_matches_torch_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = oracle.decode("bf16", codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_decode_e4m3_matches_torch_and_ocp_points():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.decode("e4m3", codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    # Points fixed by the OCP FP8 definition (E4M3: bias 7, no infinities).
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0          # largest finite
    assert got[0x08] == 2.0 ** -6                               # smallest normal
    assert got[0x01] == 2.0 ** -9                               # smallest subnormal
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])          # the only NaNs
    assert got[0x38] == 1.0 and got[0x48] == 4.0
    assert np.isnan(got).sum() == 2


def test_decode_e5m2_matches_torch_and_ocp_points():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e5m2).double().numpy()
    got = oracle.decode("e5m2", codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    # Points fixed by the OCP FP8 definition (E5M2: bias 15, IEEE-like specials).
    assert got[0x7B] == 57344.0                                 # largest finite
    assert got[0x04] == 2.0 ** -14 and got[0x01] == 2.0 ** -16  # smallest normal / subnormal
    assert got[0x7C] == np.inf and got[0xFC] == -np.inf
    assert np.isnan(got[[0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]]).all() and np.isnan(got).sum() == 6
    assert got[0x3C] == 1.0 and got[0x44] == 4.0


def test_e5m2_code_set_for_pm4_recipe():
    codes = W.e5m2_codes_in_pm4().numpy()
    allv = oracle.decode("e5m2", np.arange(256))
    inside = [c for c in range(256) if np.isfinite(allv[c]) and abs(allv[c]) <= 4.0]
    assert len(codes) == 138 and sorted(inside) == sorted(codes.tolist())


def test_e4m3_code_set_for_pm4_recipe():
    codes = W.e4m3_codes_in_pm4().numpy()
    vals = oracle.decode("e4m3", codes)
    assert len(codes) == 146
    assert np.all(np.abs(vals) <= 4.0)
    allv = oracle.decode("e4m3", np.arange(256))
    inside = [c for c in range(256) if not np.isnan(allv[c]) and abs(allv[c]) <= 4.0]
    assert sorted(inside) == sorted(codes.tolist())


# ---------------------------------------------------------------- rounding

def test_round_f16_matches_numpy():
    g = np.random.default_rng(11)
    v = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-9, 5, 20000),
                        g.uniform(-70000, 70000, 2000),
                        [0.0, -0.0, 65504.0, 65519.999, 65520.0, -65520.0, 2.0 ** -24,
                         2.0 ** -25, 3 * 2.0 ** -26, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11]])
    got = oracle.round_to("f16", v)
    ref = v.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_exact_in_f32_matches_torch():
    g = np.random.default_rng(12)
    v = (g.standard_normal(50000) * 10.0 ** g.integers(-30, 30, 50000)).astype(np.float32)
    got = oracle.round_to("bf16", v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_ties_and_no_double_rounding():
    cases = {
        1.0 + 2.0 ** -8: 1.0,                        # tie -> even (mantissa 0)
        1.0 + 3 * 2.0 ** -8: 1.0 + 2.0 ** -6,        # tie -> even (mantissa 2)
        1.0 + 2.0 ** -8 + 2.0 ** -30: 1.0 + 2.0 ** -7,  # just above the tie: rounds up
        -(1.0 + 2.0 ** -8 + 2.0 ** -30): -(1.0 + 2.0 ** -7),
    }
    for x, want in cases.items():
        code = oracle.round_to("bf16", [x])[0]
        assert oracle.decode("bf16", [code])[0] == want, x
    # overflow: halfway between the largest finite and 2^128 rounds to inf
    big = (2 - 2.0 ** -8) * 2.0 ** 127
    assert oracle.round_to("bf16", [big])[0] == 0x7F80
    assert oracle.round_to("bf16", [np.nextafter(big, 0)])[0] == 0x7F7F


def test_round_f32_matches_numpy():
    g = np.random.default_rng(13)
    v = g.standard_normal(10000) * 10.0 ** g.integers(-40, 40, 10000)
    np.testing.assert_array_equal(oracle.round_to("f32", v), v.astype(np.float32))


# ---------------------------------------------------------------- the GEMM

def _rand(shape, dt, gen, scale=1.0):
    if dt in ("e4m3", "e5m2"):
        tab = W.e4m3_codes_in_pm4() if dt == "e4m3" else W.e5m2_codes_in_pm4()
        return tab[torch.randint(0, tab.numel(), shape, generator=gen)]
    return (torch.randn(shape, generator=gen) * scale).to(W.TORCH_DTYPE[dt])


@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("a_mn,b_mn,cd_m", [(False, False, False), (True, True, True),
                                            (True, False, False), (False, True, True)])
def test_gemm_matches_numpy_float64_matmul(ab, a_mn, b_mn, cd_m):
    """Special case that reduces to a library routine: numpy's float64 matmul
    of the (exactly decoded) inputs, plus the epilogue, agrees with the oracle
    to within fp64 summation error."""
    g = torch.Generator().manual_seed(21)
    L, M, N, K = 2, 19, 23, 37
    A, B = _rand((L, M, K), ab, g), _rand((L, N, K), ab, g)
    C, X = _rand((L, M, N), "f16", g), _rand((L, M, N), "bf16", g)
    p = _problem(A, B, C, X, ab=ab, c="f16", x="bf16", a_mn=a_mn, b_mn=b_mn, cd_m=cd_m,
                 alpha=1.25, beta=-0.75, xf=3.0)
    D, Y, S = oracle.gemm(p)
    a, b, c, x = _f64(A).numpy(), _f64(B).numpy(), _f64(C).numpy(), _f64(X).numpy()
    acc = np.matmul(a, b.transpose(0, 2, 1))
    sabs = np.matmul(np.abs(a), np.abs(b).transpose(0, 2, 1))
    tol = 4 * K * 2.0 ** -53 * sabs + 1e-300
    assert np.all(np.abs(Y - acc) <= tol)
    assert np.all(np.abs(D - (1.25 * acc - 0.75 * c + 3.0 * x)) <= 2 * tol + 4 * 2.0 ** -53 * (np.abs(c) + 3 * np.abs(x)))
    np.testing.assert_allclose(S, sabs, rtol=1e-12)


def test_brute_force_fractions_8x8x16():
    """Exact rational arithmetic on an 8x8x16 problem: the oracle's fp64
    result lies within K*2^-53*sum|ab| of the exact value, and rounding the
    exact D to fp32 agrees with the oracle's rounded D."""
    g = torch.Generator().manual_seed(31)
    A = (torch.randn(1, 8, 16, generator=g)).to(torch.float16)
    B = (torch.randn(1, 8, 16, generator=g)).to(torch.float16)
    C = torch.randn(1, 8, 8, generator=g)
    p = _problem(A, B, C, ab="f16", c="f32", alpha=0.75, beta=1.5)
    D, Y, S = oracle.gemm(p)
    a = [[Fraction(float(v)) for v in row] for row in A[0].float()]
    b = [[Fraction(float(v)) for v in row] for row in B[0].float()]
    c = [[Fraction(float(v)) for v in row] for row in C[0]]
    for m in range(8):
        for n in range(8):
            acc = sum(a[m][k] * b[n][k] for k in range(16))
            d = Fraction(3, 4) * acc + Fraction(3, 2) * c[m][n]
            bound = 16 * 2.0 ** -53 * S[0, m, n]
            assert abs(Fraction(Y[0, m, n]) - acc) <= Fraction(bound) + Fraction(1, 2 ** 1070)
            assert abs(Fraction(D[0, m, n]) - d) <= Fraction(2 * bound + 2.0 ** -52 * abs(float(d)))
            # D rounded once to f32 equals the correctly rounded exact value
            assert oracle.round_to("f32", [D[0, m, n]])[0] == np.float32(float(d))


def test_integer_inputs_are_exact_config1_shape():
    """256^3 with integers in [-2,2] (the bit-exact workload): every
    intermediate is an integer or half-integer below 2^24, so the oracle's
    rounded fp32 D must equal int64 matmul arithmetic exactly."""
    w = W.WORKLOADS["int256_f16_f32"]
    inp = W.make_inputs(w)
    p = _problem(inp.A, inp.B, inp.C, ab="f16", c="f32", alpha=w.alpha, beta=w.beta)
    D, Y, _ = oracle.gemm(p)
    a = inp.A.to(torch.int64)
    b = inp.B.to(torch.int64)
    acc = torch.bmm(a, b.transpose(1, 2)).numpy()        # exact integers
    c = inp.C.to(torch.int64).numpy()                    # C integers -> exact
    d2 = 3 * acc - c                                     # 2*D = 3*acc - C
    np.testing.assert_array_equal(Y, acc)
    np.testing.assert_array_equal(D * 2, d2)
    np.testing.assert_array_equal(oracle.round_to("f32", D), (d2 / 2).astype(np.float32))


def test_identity_gives_transpose_of_B():
    g = torch.Generator().manual_seed(41)
    K = N = 24
    A = torch.eye(K, dtype=torch.float16)[None]
    B = torch.randn(1, N, K, generator=g).to(torch.float16)
    D, Y, _ = oracle.gemm(_problem(A, B, ab="f16", alpha=2.0))
    np.testing.assert_array_equal(Y[0], B[0].double().numpy().T)
    np.testing.assert_array_equal(D[0], 2.0 * B[0].double().numpy().T)


def test_closed_forms_pin_row_and_column_indices():
    M, N, K = 5, 7, 11
    ones_a = torch.ones(1, M, K, dtype=torch.float16)
    ones_b = torch.ones(1, N, K, dtype=torch.float16)
    kk = torch.arange(K, dtype=torch.float16)
    # A = 1, B(n,k) = k  ->  acc = K(K-1)/2 everywhere
    _, Y, _ = oracle.gemm(_problem(ones_a, kk.expand(1, N, K).contiguous()))
    assert np.all(Y == K * (K - 1) / 2)
    # A(m,k) = m, B = 1  ->  acc = m*K
    am = torch.arange(M, dtype=torch.float16)[None, :, None].expand(1, M, K).contiguous()
    _, Y, _ = oracle.gemm(_problem(am, ones_b))
    assert np.all(Y[0] == np.arange(M)[:, None] * K)
    # A = 1, B(n,k) = n  ->  acc = n*K
    bn = torch.arange(N, dtype=torch.float16)[None, :, None].expand(1, N, K).contiguous()
    _, Y, _ = oracle.gemm(_problem(ones_a, bn))
    assert np.all(Y[0] == np.arange(N)[None, :] * K)
    # A(m,k) = k, B(n,k) = k  ->  acc = sum k^2
    ak = kk.expand(1, M, K).contiguous()
    _, Y, _ = oracle.gemm(_problem(ak, kk.expand(1, N, K).contiguous()))
    assert np.all(Y == sum(k * k for k in range(K)))


def test_epilogue_terms_zero_alpha_zero_A():
    g = torch.Generator().manual_seed(51)
    L, M, N, K = 1, 6, 10, 8
    A = torch.randn(L, M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(L, N, K, generator=g).to(torch.bfloat16)
    C = torch.randn(L, M, N, generator=g).to(torch.float16)
    X = torch.randn(L, M, N, generator=g).to(torch.float16)
    c, x = C.double().numpy(), X.double().numpy()
    # A = 0: Y = 0 and D = beta*C + x_factor*X
    D, Y, _ = oracle.gemm(_problem(torch.zeros_like(A), B, C, X, ab="bf16", c="f16", x="f16",
                                   alpha=2.0, beta=-3.0, xf=0.5))
    assert np.all(Y == 0)
    np.testing.assert_array_equal(D, -3.0 * c + 0.5 * x)
    # alpha = 0: D does not depend on A or B
    D1, _, _ = oracle.gemm(_problem(A, B, C, X, ab="bf16", c="f16", x="f16", alpha=0.0, beta=1.0,
                                    xf=2.0))
    np.testing.assert_array_equal(D1, c + 2.0 * x)
    # beta = 0 and C full of NaN: C is not read
    Cn = torch.full_like(C, float("nan"))
    D2, Y2, _ = oracle.gemm(_problem(A, B, Cn, ab="bf16", c="f16", alpha=1.0, beta=0.0))
    assert not np.isnan(D2).any()
    np.testing.assert_array_equal(D2, Y2)
    # K = 0: acc = 0
    D3, Y3, _ = oracle.gemm(_problem(A[:, :, :0], B[:, :, :0], C, X, ab="bf16", c="f16", x="f16",
                                     alpha=5.0, beta=2.0, xf=-1.0))
    assert np.all(Y3 == 0)
    np.testing.assert_array_equal(D3, 2.0 * c - x)


def test_layout_equivalence_all_majors_and_padding():
    g = torch.Generator().manual_seed(61)
    L, M, N, K = 3, 9, 12, 20
    A = torch.randn(L, M, K, generator=g).to(torch.float16)
    B = torch.randn(L, N, K, generator=g).to(torch.float16)
    C = torch.randn(L, M, N, generator=g)
    base = oracle.gemm(_problem(A, B, C, alpha=1.5, beta=0.5))
    for a_mn in (False, True):
        for b_mn in (False, True):
            for cd_m in (False, True):
                got = oracle.gemm(_problem(A, B, C, a_mn=a_mn, b_mn=b_mn, cd_m=cd_m, alpha=1.5,
                                           beta=0.5))
                for u, v in zip(base, got):
                    np.testing.assert_array_equal(u, v)
    padded = oracle.gemm(_problem(A, B, C, alpha=1.5, beta=0.5, lda=K + 8, ldb=K + 4))
    for u, v in zip(base, padded):
        np.testing.assert_array_equal(u, v)


def test_transpose_symmetry_and_batches():
    g = torch.Generator().manual_seed(71)
    L, M, N, K = 2, 7, 13, 9
    A = torch.randn(L, M, K, generator=g).to(torch.float16)
    B = torch.randn(L, N, K, generator=g).to(torch.float16)
    C = torch.randn(L, M, N, generator=g)
    D, Y, _ = oracle.gemm(_problem(A, B, C, alpha=0.5, beta=2.0))
    Dt, Yt, _ = oracle.gemm(_problem(B, A, C.transpose(1, 2).contiguous(), alpha=0.5, beta=2.0))
    np.testing.assert_array_equal(D, Dt.transpose(0, 2, 1))
    np.testing.assert_array_equal(Y, Yt.transpose(0, 2, 1))
    for l in range(L):
        Dl, Yl, _ = oracle.gemm(_problem(A[l:l + 1], B[l:l + 1], C[l:l + 1], alpha=0.5, beta=2.0))
        np.testing.assert_array_equal(D[l], Dl[0])


def test_entries_and_row_blocks_agree_with_full():
    g = torch.Generator().manual_seed(81)
    L, M, N, K = 2, 17, 11, 33
    A = torch.randn(L, M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(L, N, K, generator=g).to(torch.bfloat16)
    X = torch.randn(L, M, N, generator=g).to(torch.bfloat16)
    p = _problem(A, B, None, X, ab="bf16", x="bf16", cd_m=True, alpha=1.0, xf=-2.0)
    D, Y, S = oracle.gemm(p)
    rng = np.random.default_rng(3)
    ms, ns, ls = rng.integers(0, M, 50), rng.integers(0, N, 50), rng.integers(0, L, 50)
    De, Ye, Se = oracle.gemm_entries(p, ms, ns, ls)
    np.testing.assert_array_equal(De, D[ls, ms, ns])
    np.testing.assert_array_equal(Ye, Y[ls, ms, ns])
    np.testing.assert_array_equal(Se, S[ls, ms, ns])
    Dr, Yr, _ = oracle.gemm_rows(p, 5, 12)
    np.testing.assert_array_equal(Dr, D[:, 5:12])


@pytest.mark.parametrize("a_dt,b_dt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_fp8_pairs_match_numpy_float64_matmul(a_dt, b_dt):
    """E5M2 and mixed E4M3 x E5M2 operands: numpy float64 matmul of the exact
    values (decoded by torch) agrees with the oracle within fp64 error."""
    g = torch.Generator().manual_seed(91)
    L, M, N, K = 2, 17, 21, 40
    A, B = _rand((L, M, K), a_dt, g), _rand((L, N, K), b_dt, g)
    C = _rand((L, M, N), "f16", g)
    p = _problem(A, B, C, ab=a_dt, b=b_dt, c="f16", b_mn=True, alpha=0.25, beta=1.0)
    D, Y, S = oracle.gemm(p)
    a, b = _f64(A, a_dt).numpy(), _f64(B, b_dt).numpy()
    acc = np.matmul(a, b.transpose(0, 2, 1))
    tol = 4 * K * 2.0 ** -53 * np.matmul(np.abs(a), np.abs(b).transpose(0, 2, 1)) + 1e-300
    assert np.all(np.abs(Y - acc) <= tol)
    assert np.all(np.abs(D - (0.25 * acc + C.double().numpy())) <= 2 * tol + 1e-12)


def test_relu_variant_closed_forms_and_numpy():
    """relu(alpha*acc + beta*C) + x_factor*X, the rectifier before X is added
    ("custom_epilogue_dense_gemm.py", epilogue() function)."""
    g = torch.Generator().manual_seed(93)
    L, M, N, K = 1, 12, 10, 16
    A = torch.randn(L, M, K, generator=g).to(torch.float16)
    B = torch.randn(L, N, K, generator=g).to(torch.float16)
    C = torch.randn(L, M, N, generator=g).to(torch.float16)
    X = torch.randn(L, M, N, generator=g).to(torch.float16)
    c, x = C.double().numpy(), X.double().numpy()
    # A = 0: D = max(beta*C, 0) + x_factor*X exactly
    D0, Y0, _ = oracle.gemm(_problem(torch.zeros_like(A), B, C, X, c="f16", x="f16", alpha=1.0,
                                     beta=-2.0, xf=0.5, relu=True))
    np.testing.assert_array_equal(D0, np.maximum(-2.0 * c, 0.0) + 0.5 * x)
    assert np.all(Y0 == 0)
    # general: numpy float64
    D, Y, S = oracle.gemm(_problem(A, B, C, X, c="f16", x="f16", alpha=1.5, beta=0.5, xf=-1.0,
                                   relu=True))
    acc = np.matmul(A.double().numpy(), B.double().numpy().transpose(0, 2, 1))
    want = np.maximum(1.5 * acc + 0.5 * c, 0.0) - x
    assert np.all(np.abs(D - want) <= 8 * K * 2.0 ** -53 * (S + np.abs(c) + np.abs(x)))
    # the same problem without relu differs exactly where alpha*acc + beta*C < 0
    Dl, _, _ = oracle.gemm(_problem(A, B, C, X, c="f16", x="f16", alpha=1.5, beta=0.5, xf=-1.0))
    neg = (1.5 * acc + 0.5 * c) < 0
    assert neg.any() and (~neg).any()
    np.testing.assert_array_equal(D[~neg], Dl[~neg])
    assert np.all(D[neg] == -x[neg])


def test_tf32_storage_decodes_as_fp32_and_generator_rounds_to_tf32():
    g = torch.Generator().manual_seed(95)
    v = torch.randn(4096, generator=g) * 10.0 ** torch.randint(-20, 20, (4096,), generator=g)
    r = W.round_to_tf32(v)
    bits = r.view(torch.int32)
    assert torch.all((bits & 0x1FFF) == 0)                     # 10 fraction bits left
    # nearest: within half a tf32 spacing, ties (constructed) to even
    e = torch.floor(torch.log2(v.abs().double()))
    half = torch.exp2(e - 11)
    assert torch.all((r.double() - v.double()).abs() <= half)
    ties = torch.tensor([1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11], dtype=torch.float32)
    assert W.round_to_tf32(ties).tolist() == [1.0, 1.0 + 2.0 ** -9]
    codes = bits.numpy().view(np.uint32)[:64]
    np.testing.assert_array_equal(oracle.decode("tf32", codes), oracle.decode("f32", codes))


# ---------------------------------------------------------------- half-precision accumulator term

def test_partial_sum_term_brute_force_fractions():
    """P = sum over the chunk boundaries (every 16 k and k = K) of |exact
    running sum|, checked against exact rational arithmetic on a K that is
    not a multiple of the chunk (50 = 3*16 + 2), for two chunk sizes."""
    g = torch.Generator().manual_seed(37)
    A = torch.randn(1, 4, 50, generator=g).to(torch.float16)
    B = torch.randn(1, 3, 50, generator=g).to(torch.float16)
    a = [[Fraction(float(v)) for v in row] for row in A[0].float()]
    b = [[Fraction(float(v)) for v in row] for row in B[0].float()]
    for chunk, bounds in ((16, (16, 32, 48, 50)), (32, (32, 50))):
        D, Y, S, P = oracle.gemm(_problem(A, B, ab="f16", alpha=1.0, acc_chunk=chunk))
        for m in range(4):
            for n in range(3):
                exact = sum(abs(sum(a[m][k] * b[n][k] for k in range(e))) for e in bounds)
                assert abs(Fraction(P[0, m, n]) - exact) <= Fraction(1e-12) * (1 + exact)


def test_partial_sum_term_closed_forms():
    """All-ones A and B: the running sum after k terms is k, so P is the sum
    of the boundaries themselves (16+32+48+64 = 160 for K = 64, chunk 16;
    32+64+70 = 166 for K = 70, chunk 32).  Signs alternating along k make
    every even running sum 0: with chunk 2, P = 0 exactly; with chunk 3 the
    boundaries 3, 6, ... alternate |1| and |0|."""
    for K, chunk, want in ((64, 16, 160.0), (70, 32, 166.0), (1, 16, 1.0)):
        A = torch.ones(1, 2, K, dtype=torch.float16)
        B = torch.ones(1, 2, K, dtype=torch.float16)
        _, Y, _, P = oracle.gemm(_problem(A, B, ab="f16", alpha=1.0, acc_chunk=chunk))
        assert np.all(P == want) and np.all(Y == K)
    K = 12
    alt = torch.tensor([(-1.0) ** k for k in range(K)], dtype=torch.float16)
    A = alt.expand(1, 2, K).contiguous()
    B = torch.ones(1, 2, K, dtype=torch.float16)
    _, _, _, P2 = oracle.gemm(_problem(A, B, ab="f16", alpha=1.0, acc_chunk=2))
    _, _, _, P3 = oracle.gemm(_problem(A, B, ab="f16", alpha=1.0, acc_chunk=3))
    assert np.all(P2 == 0.0)
    assert np.all(P3 == 2.0)       # boundaries 3, 6, 9, 12: |1|, |0|, |1|, |0|


def test_partial_sum_term_layouts_entries_and_off():
    """P does not depend on layouts, entries and row blocks agree with the
    full problem, acc_chunk = 0 returns the three-array result, and a
    negative chunk is rejected."""
    g = torch.Generator().manual_seed(41)
    A = torch.randn(2, 9, 40, generator=g).to(torch.bfloat16)
    B = torch.randn(2, 7, 40, generator=g).to(torch.bfloat16)
    base = oracle.gemm(_problem(A, B, ab="bf16", alpha=1.0, acc_chunk=16))
    assert len(base) == 4 and np.all(base[3] >= np.abs(base[1]))
    alt = _problem(A, B, ab="bf16", a_mn=True, b_mn=True, alpha=1.0, acc_chunk=16)
    np.testing.assert_array_equal(oracle.gemm(alt)[3], base[3])
    ms, ns, ls = np.array([0, 8, 4]), np.array([6, 0, 3]), np.array([1, 0, 1])
    pe = oracle.gemm_entries(alt, ms, ns, ls)[3]
    np.testing.assert_array_equal(pe, base[3][ls, ms, ns])
    np.testing.assert_array_equal(oracle.gemm_rows(alt, 2, 5)[3], base[3][:, 2:5])
    assert len(oracle.gemm(_problem(A, B, ab="bf16", alpha=1.0))) == 3
    with pytest.raises(ValueError):
        oracle.gemm(_problem(A, B, ab="bf16", alpha=1.0, acc_chunk=-1))

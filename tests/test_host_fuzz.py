"""Property-based robustness of the host-only C ABI calls (CPU): for arbitrary
arguments gemm_check and gemm_plan return a defined status, never crash, and
every accepted problem gets a configuration consistent with it."""
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st

import dense_gemm_epilogue_persistent_gb300 as G

STATUSES = {G.GEMM_OK, G.GEMM_ERR_INVALID_ARG, G.GEMM_ERR_UNSUPPORTED_DTYPE,
            G.GEMM_ERR_MISALIGNED, G.GEMM_ERR_UNSUPPORTED_CONFIG}
TYPES = ["f32", "f16", "bf16", "e4m3", "e5m2", "tf32"]

dims = st.one_of(st.integers(-2, 4), st.integers(0, 20000), st.sampled_from([1, 8, 16, 128, 4096]))
ptrs = st.one_of(st.none(), st.sampled_from([1 << 20, (1 << 20) + 8, (1 << 20) + 16, 1 << 30]))


@settings(max_examples=400, deadline=None)
@given(M=dims, N=dims, K=dims, L=st.integers(-1, 4), lda=dims, ldb=dims,
       la=st.integers(-1, 2), lb=st.integers(-1, 2), cdm=st.integers(-1, 2),
       ab=st.sampled_from(TYPES + [7]), b=st.sampled_from([None] + TYPES),
       c=st.sampled_from(TYPES), d=st.sampled_from(TYPES), x=st.sampled_from(TYPES),
       y=st.sampled_from(TYPES), epi=st.integers(-1, 2), acc=st.sampled_from(TYPES),
       A=ptrs, B=ptrs, C=ptrs, X=ptrs, D=ptrs, Y=ptrs,
       alpha=st.sampled_from([0.0, 1.0, -2.5]), beta=st.sampled_from([0.0, 1.0]),
       xf=st.sampled_from([0.0, 3.0]))
def test_check_and_plan_never_crash(M, N, K, L, lda, ldb, la, lb, cdm, ab, b, c, d, x, y, epi,
                                    acc, A, B, C, X, D, Y, alpha, beta, xf):
    code = lambda t: G.DTYPE_CODES[t] if isinstance(t, str) else int(t)
    dt = G.gemm_dtypes_t(code(ab), code(c), code(d), code(x), code(y), cdm,
                         0 if b is None else code(b), epi, code(acc))
    p = G.make_problem(M, N, K, L, A, lda, la, B, ldb, lb, C, X, D, Y, alpha, beta, xf, dt)
    st_check = G.gemm_check(p)
    assert st_check in STATUSES
    st_plan, cfg = G.gemm_plan(p, 152, 232448)
    if st_check != G.GEMM_OK:
        assert st_plan == st_check                   # the planner validates first
        return
    if M == 0 or N == 0 or L == 0:
        return
    assert st_plan in (G.GEMM_OK, G.GEMM_ERR_UNSUPPORTED_CONFIG)
    if st_plan == G.GEMM_OK:
        assert cfg.cta_group in (1, 2) and cfg.tile_n in (128, 256) and cfg.cluster_m in (1, 2)
        rows = cfg.tile_m * cfg.cluster_m
        assert cfg.tiles == (-(-M // rows)) * (-(-N // cfg.tile_n)) * L
        assert 2 <= cfg.stages and 2 <= cfg.epi_slots <= 6 and cfg.smem_bytes <= 232448
        assert 0 <= cfg.tail_split <= cfg.tiles
        assert 0 < cfg.grid_ctas <= 152 * cfg.cta_group * cfg.cluster_m

"""The device watchdog, exercised without faulting or hanging the GPU.

Every mbarrier wait in the kernel is bounded.  A test-only configuration
(inject_stall) makes the MMA warp wait on a barrier that nothing ever arrives
at: every role must then give up after the configured limit, drain, free its
tensor memory and return, leaving GEMM_ERR_DEVICE_TIMEOUT (role 6) in the
status word -- and the context must stay usable for the next, normal GEMM.
"""
import pytest
import torch

import dense_gemm_epilogue_persistent_gb300 as G
from gemm_cases import Case, compare_full, prepare, run_gpu

pytestmark = pytest.mark.gpu

# (cta_group, tile_n, cluster_m, cluster_n, epi_warps, stream_k): single CTAs,
# pairs, clusters sharing B, A or both through multicast, eight epilogue
# warps, and stream-K (whose owners also wait for partial sums)
VARIANTS = [(1, 256, 1, 1, 1, 0), (2, 256, 1, 1, 1, 0), (2, 256, 2, 1, 1, 0),
            (1, 128, 2, 1, 1, 0), (2, 256, 1, 2, 1, 0), (2, 160, 2, 2, 1, 0),
            (1, 128, 1, 1, 2, 0), (2, 256, 1, 1, 2, 0), (1, 256, 1, 1, 2, 2), (2, 128, 1, 1, 1, 2)]


@pytest.mark.parametrize("variant", VARIANTS)
def test_injected_stall_times_out_cleanly_and_context_survives(variant):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g = G.Gemm(0)
    try:
        case = Case(M=1024, N=768, K=512, L=1, ab="f16", c="f16", d="f16", x="f16", y="f16",
                    alpha=1.0, beta=1.0, xf=1.0, seed=77)
        prep = prepare(case)
        cg, bn, mc, nc, epw, sk = variant
        G.gemm_set_timeout_ns(g.handle, 50_000_000)           # 50 ms per wait
        g.set_config(G.gemm_config_t(cta_group=cg, tile_n=bn, cluster_m=mc, cluster_n=nc,
                                     epi_warps=epw, stream_k=sk, inject_stall=1))
        run_gpu(g, prep)
        st, detail = g.sync_status()
        assert st == G.GEMM_ERR_DEVICE_TIMEOUT
        assert detail >> 24 == 0xE0 and (detail >> 16) & 0xFF == 6, hex(detail)
        st, detail = g.sync_status()                             # cleared by the read
        assert st == G.GEMM_OK and detail == 0
        # the same handle, stream and context run a normal GEMM correctly
        G.gemm_set_timeout_ns(g.handle, 0)
        g.set_config(G.gemm_config_t(cta_group=cg, tile_n=bn, cluster_m=mc, cluster_n=nc,
                                     epi_warps=epw, stream_k=sk))
        D, Y = run_gpu(g, prep)
        st, detail = g.sync_status()
        assert st == G.GEMM_OK, hex(detail)
        assert (g.last_config().stream_k > 0) == (sk == 2)
        compare_full(prep, D, Y)
    finally:
        g.close()

"""Forced configuration fields reach the launch: group_m and the L2 hints set
through gemm_set_config are the ones gemm_last_config reports, and every run
ends with a clean device status and a result equal to the automatic one."""
import pytest
import torch

import workloads as W
import dense_gemm_epilogue_persistent_gb300 as G
from gemm_cases import Case, prepare, run_gpu

pytestmark = pytest.mark.gpu


def test_forced_group_m_and_l2_hints_reach_the_launch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g = G.Gemm(0)
    try:
        prep = prepare(Case(M=1024, N=1024, K=256, L=1, ab="bf16", c="f32", d="f32",
                            alpha=1.0, beta=1.0, dist="int2", seed=11))
        D_auto, _ = run_gpu(g, prep)
        assert g.sync_status()[0] == G.GEMM_OK
        for gm in (2, 4):
            g.set_config(group_m=gm)
            D, _ = run_gpu(g, prep)
            assert g.sync_status()[0] == G.GEMM_OK
            assert g.last_config().group_m == gm
            assert torch.equal(D, D_auto)
        g.set_config(l2_hints=0x100 | 0x2A)
        D, _ = run_gpu(g, prep)
        assert g.sync_status()[0] == G.GEMM_OK
        assert g.last_config().l2_hints == 0x2A
        assert torch.equal(D, D_auto)
    finally:
        g.close()

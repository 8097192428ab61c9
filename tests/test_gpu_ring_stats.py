"""The ring-statistics build (per-role wait counters compiled into a separate
library) and its report tool, run in a subprocess so that the test process
keeps the product library: the counters must account for exactly the stages
and epilogue chunks the launch geometry implies, and every wait share must be
a fraction of its role's loop."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ring_stats_tool_accounts_for_every_stage_and_chunk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "ring_stats.py",
                        "int256_f16_f32", "gemm2048_bf16_f32", "ragged_e4m3_f16",
                        "--launches", "5", "--json"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    rows = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert [x["workload"] for x in rows] == ["int256_f16_f32", "gemm2048_bf16_f32",
                                             "ragged_e4m3_f16"]
    for x in rows:
        items = x["tiles"] + x["tail_split"]
        assert x["stages"] == items * x["k_blocks"], x
        whole, halves = x["tiles"] - x["tail_split"], 2 * x["tail_split"]
        assert x["chunks"] == x["cta_group"] * (whole * x["tile_n"] // 32 +
                                                halves * x["tile_n"] // 64), x
        for k in ("mma_wait_stage_pct", "mma_wait_accumulator_pct", "producer_wait_drain_pct",
                  "epilogue_wait_accumulator_pct", "epilogue_wait_cx_pct"):
            assert 0.0 <= x[k] <= 100.0, (k, x)
        assert x["cycles_per_stage"] > 0

"""The configuration runner: forced group_m values reach the launch and every
run ends with a clean device status."""
import json

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_tune_runs_forced_group_m(capsys):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_epilogue_persistent_gb300 import tune
    assert tune.main(["gemm2048_bf16_f32", "--group-m", "2,4", "--launches", "3"]) == 0
    rows = [json.loads(l) for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert [r["group_m"] for r in rows] == [2, 4]
    assert all(r["tflops"] > 0 for r in rows)
    assert tune.main(["int256_f16_f32", "--once", "--l2-hints", "0x2a"]) == 0
    row = json.loads(capsys.readouterr().out.splitlines()[-1])
    assert row["l2_hints"] == 0x2A and "us" not in row

"""The N > 1 path of bench.py on the CPU: world-size-2 gloo ranks.

The GEMM shards as independent replicas (no data-path collective); the only
multi-rank logic is the barrier, the max-over-ranks time and the whole-job
throughput, plus the reference arm's rule that only rank 0 runs and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    pg = bench.init_ranks(world, rank)
    pg.barrier()
    m = bench.max_over_ranks(times[rank], pg)
    v = bench.whole_job_tflops(1e12, 10, world, m)
    out.put((rank, m, v))
    pg.barrier()
    pg.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world, port = 2, _free_port()
    times = [12.5, 20.0]                       # ms: rank 1 is the slow one
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 20.0                       # every rank sees the slowest time
        assert v == pytest.approx(1e12 * 10 * 2 / 0.020 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.init_ranks(1, 0) is None
    assert bench.max_over_ranks(3.0, None) == 3.0
    assert bench.whole_job_tflops(2e12, 5, 1, 1000.0) == pytest.approx(10.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--workload", "int256_f16_f32",
                        "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 1:
        assert lines == []
    else:
        d = json.loads(lines[-1])
        assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
        assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
        assert d["n_gpus"] == 2

"""Per-role pipeline statistics of the GEMM kernel on a workload.

    python ring_stats.py [WORKLOAD ...] [--launches N] [--json]

Builds (if needed) and loads the ring-statistics library -- the product
sources compiled with per-role wait counters -- runs each named workload
(default: the 8192^3 fp16 custom-epilogue GEMM) back to back N times and
reports, for the last launch, the share of each role's loop spent waiting:

  MMA issuer   waiting for a stage to land (the operand feed) and for a free
               accumulator stage (the epilogue), and cycles per ring stage;
  producer     waiting for a stage to drain (a full ring);
  epilogue     waiting for a finished accumulator and for C/X to land.

A measurement tool beside bench.py: it draws the workloads' inputs with
workloads.py, as the benchmark does.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from dense_gemm_epilogue_persistent_gb300 import build as _build  # noqa: E402


def _device_inputs(G, W, w, torch):
    inp = W.make_inputs(w)
    dev = torch.device("cuda")
    A = W.to_storage(inp.A, w.a_mn_major).to(dev)
    B = W.to_storage(inp.B, w.b_mn_major).to(dev)
    C = W.to_storage(inp.C, w.cd_m_major).to(dev) if inp.C is not None else None
    X = W.to_storage(inp.X, w.cd_m_major).to(dev) if inp.X is not None else None
    shape = (w.L, w.N, w.M) if w.cd_m_major else (w.L, w.M, w.N)
    D = torch.empty(shape, dtype=W.TORCH_DTYPE[w.d], device=dev)
    Y = torch.empty(shape, dtype=W.TORCH_DTYPE[w.y], device=dev) if w.y else None
    dt = G.make_dtypes(w.ab, w.c or "f32", w.d, w.x or "f32", w.y or "f32",
                       G.GEMM_MN_MAJOR if w.cd_m_major else G.GEMM_K_MAJOR, b=w.b,
                       epilogue=G.GEMM_EPI_RELU if w.relu else G.GEMM_EPI_LINEAR, acc=w.acc)
    return A, B, C, X, D, Y, dt


def measure(names, launches=30, config=None):
    """Run each workload `launches` times with the statistics library (and a
    forced configuration, if given: gemm_config_t fields); return one summary
    dict per workload."""
    import dense_gemm_epilogue_persistent_gb300 as G
    G.select_library(_build.build(ring_stats=True))
    import torch
    import workloads as W
    g = G.Gemm(0)
    if config:
        g.set_config(G.gemm_config_t(**config))
    out = []
    try:
        for name in names:
            w = W.WORKLOADS[name]
            A, B, C, X, D, Y, dt = _device_inputs(G, W, w, torch)
            run = lambda: g.run(w.M, w.N, w.K, w.L, A, A.shape[-1], int(w.a_mn_major), B,
                                B.shape[-1], int(w.b_mn_major), C, X, D, Y, w.alpha, w.beta,
                                w.x_factor, dt)
            run()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(launches):
                run()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / launches
            st, detail = g.sync_status()
            if st != G.GEMM_OK:
                raise RuntimeError(f"{name}: {G.gemm_status_string(st)} {detail:#x}")
            cfg = g.last_config()
            rows = g.ring_stats()
            mma = [r for r in rows if r[3] > 0]             # CTAs that issue MMAs
            share = lambda rs, i, j: sum(r[i] for r in rs) / max(1, sum(r[j] for r in rs))
            out.append({
                "workload": name,
                "kernel": f"{cfg.tile_m}x{cfg.tile_n} cta_group={cfg.cta_group} "
                          f"cluster_m={cfg.cluster_m} cluster_n={cfg.cluster_n} "
                          f"stages={cfg.stages} "
                          f"epi_slots={cfg.epi_slots} epi_warps={cfg.epi_warps} "
                          f"grid={cfg.grid_ctas}",
                "tflops_with_counters": round(w.flops / ms / 1e9, 1),
                "mma_wait_stage_pct": round(100 * share(mma, 0, 2), 2),
                "mma_wait_accumulator_pct": round(100 * share(mma, 1, 2), 2),
                "cycles_per_stage": round(sum(r[2] for r in mma) / max(1, sum(r[3] for r in mma)), 1),
                "producer_wait_drain_pct": round(100 * share(rows, 4, 5), 2),
                "epilogue_wait_accumulator_pct": round(100 * share(rows, 6, 8), 2),
                "epilogue_wait_cx_pct": round(100 * share(rows, 7, 8), 2),
                "epilogue_read_cycles_per_chunk": round(share(rows, 10, 13), 1),
                "epilogue_math_cycles_per_chunk": round(share(rows, 11, 13), 1),
                "epilogue_issue_cycles_per_chunk": round(share(rows, 12, 13), 1),
                "epilogue_cx_wait_cycles_per_chunk": round(share(rows, 7, 13), 1),
                "stages": int(sum(r[3] for r in mma)),
                "chunks": int(sum(r[9] for r in rows)),
                "tiles": int(cfg.tiles), "tail_split": int(cfg.tail_split),
                "tile_n": int(cfg.tile_n), "cta_group": int(cfg.cta_group),
                "k_blocks": -(-w.K // cfg.tile_k),
            })
            del A, B, C, X, D, Y
    finally:
        g.close()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("workloads", nargs="*", default=["efc8192_f16"])
    ap.add_argument("--launches", type=int, default=30)
    ap.add_argument("--json", action="store_true")
    ap.add_argument("--config", default="", help="forced configuration, e.g. cta_group=2,tile_n=256")
    args = ap.parse_args(argv)
    config = {}
    for kv in filter(None, args.config.split(",")):
        k, v = kv.split("=")
        config[k] = int(v, 0)
    res = measure(args.workloads, args.launches, config)
    for r in res:
        print(json.dumps(r) if args.json else
              f"{r['workload']}: {r['kernel']}  {r['tflops_with_counters']} TFLOP/s | MMA waits: "
              f"stage {r['mma_wait_stage_pct']}%, accumulator {r['mma_wait_accumulator_pct']}%, "
              f"{r['cycles_per_stage']} cycles/stage | producer waits for drain "
              f"{r['producer_wait_drain_pct']}% | epilogue waits: accumulator "
              f"{r['epilogue_wait_accumulator_pct']}%, C/X {r['epilogue_wait_cx_pct']}%")
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Run a workload under forced launch configurations.

    python -m dense_gemm_epilogue_persistent_gb300.tune WORKLOAD [--group-m 4,8,12]
        [--l2-hints 42,40] [--cta-group N] [--tile-n N] [--stages 2,3]
        [--epi-slots 2,4] [--epi-wait-ns 0,1000] [--launches N] [--once]

For each combination of the listed group_m, l2_hints, stages, epi_slots and
epi_wait_ns values (absent: automatic; other fields automatic unless given) it runs the workload back to back `--launches` times
and prints TFLOP/s from CUDA events; with --once it runs exactly one launch per
configuration and times nothing, for a profiler capturing one launch of each
(e.g. ncu -k regex:persistent).  Run from the repository root (it reads the
workload definitions there).
"""
from __future__ import annotations

import argparse
import itertools
import json
import sys

from .ring_stats import _device_inputs


def _ints(s: str | None):
    return [int(x, 0) for x in s.split(",")] if s else [0]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("workload")
    ap.add_argument("--group-m", default=None)
    ap.add_argument("--l2-hints", default=None,
                    help="2 bits each: A/B loads, C/X loads, D/Y stores (0 normal, 1 last, "
                         "2 first); 0 = automatic, 0x100 = all normal")
    ap.add_argument("--cta-group", type=int, default=0)
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--stages", default=None)
    ap.add_argument("--epi-slots", default=None)
    ap.add_argument("--epi-wait-ns", default=None,
                    help="suspend hint of the epilogue's accumulator wait (0 = none)")
    ap.add_argument("--launches", type=int, default=200)
    ap.add_argument("--once", action="store_true")
    args = ap.parse_args(argv)

    sys.path.insert(0, ".")
    import torch
    import workloads as W
    import dense_gemm_epilogue_persistent_gb300 as G

    w = W.WORKLOADS[args.workload]
    g = G.Gemm(0)
    A, B, C, X, D, Y, dt = _device_inputs(G, W, w, torch)

    def run():
        g.run(w.M, w.N, w.K, w.L, A, A.shape[-1], int(w.a_mn_major), B, B.shape[-1],
              int(w.b_mn_major), C, X, D, Y, w.alpha, w.beta, w.x_factor, dt)

    waits = [None] if args.epi_wait_ns is None else _ints(args.epi_wait_ns)
    for gm, l2, st, es, ew in itertools.product(_ints(args.group_m), _ints(args.l2_hints),
                                                _ints(args.stages), _ints(args.epi_slots), waits):
        g.set_config(G.gemm_config_t(cta_group=args.cta_group, tile_n=args.tile_n, group_m=gm,
                                     l2_hints=(l2 | 0x100) if l2 else 0, stages=st,
                                     epi_slots=es, epi_wait_ns=0 if ew is None else ew + 1))
        out = {"workload": args.workload}
        if args.once:
            run()
            torch.cuda.synchronize()
        else:
            for _ in range(10):
                run()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(args.launches):
                run()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.launches
            out.update(us=round(ms * 1e3, 2), tflops=round(w.flops / ms / 1e9, 1))
        st, detail = g.sync_status()
        if st != G.GEMM_OK:
            raise RuntimeError(f"{G.gemm_status_string(st)} {detail:#x}")
        cfg = g.last_config()
        out.update(group_m=cfg.group_m, l2_hints=cfg.l2_hints, epi_wait_ns=cfg.epi_wait_ns,
                   cta_group=cfg.cta_group,
                   tile_n=cfg.tile_n, stages=cfg.stages, epi_slots=cfg.epi_slots)
        print(json.dumps(out), flush=True)
    g.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())

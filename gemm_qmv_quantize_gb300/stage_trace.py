"""Per-stage timeline of a Q4_0 / Q4_K decode stack (the streaming kernel, M = 1..4).

Builds the library with -DQMV_STAGE_TRACE into _build/libqmv_trace.so (the product
library is untouched), runs one workload of bench.py as bench.py runs it (CUDA graph,
launch overlap on) and prints, per kind of stage, where a stage's time goes:

  release    from the previous launch's last warp to this launch's programmatic-
             dependency wait returning (first CTA .. last CTA)
  prologue   from the wait to the activation prologue's CTA barrier (x loaded,
             quantized to Q8_1, staged)
  first      from that barrier to the first weight chunk of the median warp landing
  body       from that barrier to the last warp's end
  tail       last warp's end minus the median warp's end
  late CTA   how far the last CTA's end trails the median CTA's
  ideal      the stage's algorithmic bytes at 7.2 TB/s (a read-only stream's rate)

  python -m gemm_qmv_quantize_gb300.stage_trace [--workload llama2_7b_q4_0_m1] [--json out.json]

Times come from %globaltimer (whose resolution on a GB300 is 32 ns to 1 us:
averages over the stages are meaningful, single stamps are coarse).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STAGE_KINDS = {"llama2_7b_q4_0_m1": ["qkv", "o", "gate_up", "down"], "qwen3_8b_q4_k_m1": ["qkv", "o", "gate_up", "down"]}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="llama2_7b_q4_0_m1")
    ap.add_argument("--replays", type=int, default=20, help="untimed graph replays before the traced one")
    ap.add_argument("--json", default=None, help="also write the per-stage rows to this file")
    args = ap.parse_args(argv)
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import numpy as np
    import torch

    from gemm_qmv_quantize_gb300 import _binding, build
    lib_path = build.build(defines=("QMV_STAGE_TRACE",), name="libqmv_trace.so")
    _binding._LIB_PATH = lib_path   # this process calls the traced build
    import bench
    import gemm_qmv_quantize_gb300 as q
    L = q.lib()
    L.qmv_stage_trace_set.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    L.qmv_stage_trace_set.restype = None

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stack = bench.Stack(args.workload, dev)
    n = len(stack.stages)
    ctas, warps, fields = 152 * 4, 16, 8
    rec = torch.zeros(n * ctas * warps * fields, dtype=torch.int64, device=dev)
    q.set_launch_overlap(True)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        stack.run()
        torch.cuda.synchronize()
        L.qmv_stage_trace_set(rec.data_ptr(), n, ctas)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            stack.run()
        L.qmv_stage_trace_set(None, 0, 0)
        for _ in range(args.replays):
            graph.replay()
        torch.cuda.synchronize()
        rec.zero_()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
    torch.cuda.synchronize()
    step_us = a.elapsed_time(b) * 1e3
    t = rec.cpu().numpy().reshape(n, ctas, warps, fields).astype(np.float64)
    live = t[..., 7] > 0
    rows = []
    for i in range(n):
        lv = live[i]

        def per_cta(k, fn):
            v = np.where(lv, t[i][..., k], np.nan)
            with np.errstate(all="ignore"):
                out = fn(v, axis=1)
            return out[~np.isnan(out)]
        end_w = t[i][..., 4][lv]
        rows.append(dict(
            stage=i, mbytes=stack.launch_bytes(stack.stages[i]) / 1e6,
            rel_min=per_cta(1, np.nanmin).min(), rel_max=per_cta(1, np.nanmax).max(),
            sync_med=float(np.median(t[i][..., 2][lv])), first_med=float(np.median(t[i][..., 3][lv])),
            end_med=float(np.median(end_w)), end_max=float(end_w.max()),
            cta_end_med=float(np.median(per_cta(4, np.nanmax))), cta_end_max=float(per_cta(4, np.nanmax).max())))
    kinds = STAGE_KINDS.get(args.workload)
    summary = {}
    for r in rows[1:]:
        i = r["stage"]
        kind = "lm_head" if (kinds and i == n - 1) else (kinds[i % len(kinds)] if kinds else "stage")
        prev = rows[i - 1]
        d = dict(release_first=(r["rel_min"] - prev["end_max"]) / 1e3, release_last=(r["rel_max"] - prev["end_max"]) / 1e3,
                 prologue=(r["sync_med"] - r["rel_max"]) / 1e3, first=(r["first_med"] - r["sync_med"]) / 1e3,
                 body=(r["end_max"] - r["sync_med"]) / 1e3, tail=(r["end_max"] - r["end_med"]) / 1e3,
                 late_cta=(r["cta_end_max"] - r["cta_end_med"]) / 1e3, stage=(r["end_max"] - prev["end_max"]) / 1e3,
                 ideal=r["mbytes"] * 1e6 / 7.2e12 * 1e6)
        summary.setdefault(kind, []).append(d)
    print(f"{args.workload}: {n} launches, traced step {step_us:.1f} us, "
          f"{stack.bytes_per_step / step_us / 1e3:.1f} GB/s (the traced build is a little slower than the product)")
    cols = ["stage", "ideal", "release_first", "release_last", "prologue", "first", "body", "tail", "late_cta"]
    print(f"{'kind':8s} {'n':>3s} " + " ".join(f"{c:>13s}" for c in cols) + "   (us, mean over the kind's stages)")
    for kind, ds in summary.items():
        print(f"{kind:8s} {len(ds):3d} " + " ".join(f"{statistics.mean(d[c] for d in ds):13.3f}" for c in cols))
    if args.json:
        with open(args.json, "w") as f:
            json.dump(dict(workload=args.workload, step_us=step_us, summary={k: {c: statistics.mean(d[c] for d in v)
                                                                                  for c in cols} for k, v in summary.items()}),
                      f, indent=1)


if __name__ == "__main__":
    main()

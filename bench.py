#!/usr/bin/env python3
"""Benchmark of the weight-only-quantized skinny matmul hot path on GB300.

Default workload: the Llama-2-7B-shaped Q4_0 decode stack at M = 1 -- 32 layers of
{q, k, v, o 4096x4096; gate, up 11008x4096; down 4096x11008} plus the 32000x4096
lm_head, 225 matrices, 3,716,481,024 bytes of Q4_0 weights, each call quantizing a
fresh fp32 activation row to Q8_1 and running the Q4_0 x Q8_1 MMVQ ("Machine
Learning on NVIDIA CMP", section "llama.cpp results": Llama-2-7B-Q4_0 decode). One
step = one pass over the stack = one decoded token. Calls run in stream order
(each waits for the previous one, as in decode), captured once in a CUDA graph.

metric: achieved weight-stream GB/s (bytes = packed weights + scales + Q8_1
activations + fp32 outputs, per step) and its fraction of the measured HBM copy
bandwidth; tok/s equivalent = M / step time.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--eager]
Under torchrun every rank runs an independent replica (the path has no exchange
step); the value is the units all ranks processed / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved weight-stream GB/s and % of HBM roofline; equiv. decode tok/s (M=1..8)"
FALLBACK_HBM_GBS = 6800.0
Q4_0_BLOCK, Q4_K_BLOCK, Q8_1_BLOCK = 18, 144, 36

# ----------------------------------------------------------------------------- workloads


def llama2_7b_stack():
    layer = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
    return [("q4_0", n, k) for _ in range(32) for (n, k) in layer] + [("q4_0", 32000, 4096)]


def llama2_7b_stages():
    """Decode dependency structure: per layer {q, k, v} read the layer input, o reads
    attention's output, {gate, up} read the MLP input, down reads their product;
    then the lm_head. 129 dependent stages for 225 matrices."""
    st = []
    for layer in range(32):
        b = 7 * layer
        st += [[b, b + 1, b + 2], [b + 3], [b + 4, b + 5], [b + 6]]
    return st + [[224]]


def dense_27b_stack(mixed: bool, layers: int = 64):
    """64 layers of {qkv 7168x5120, o 5120x5120, gate/up 17408x5120, down 5120x17408};
    mixed: attention projections of layers 3, 7, ..., 63 in FP8, plus an NVFP4 lm_head.
    `layers` < 64 gives the first layers of the same stack (and its lm_head)."""
    mats = []
    for layer in range(layers):
        attn = "fp8" if (mixed and layer % 4 == 3) else "nvfp4"
        mats += [(attn, 7168, 5120), (attn, 5120, 5120), ("nvfp4", 17408, 5120), ("nvfp4", 17408, 5120),
                 ("nvfp4", 5120, 17408)]
    if mixed:
        mats.append(("nvfp4", 151936, 5120))
    return mats


def dense_27b_stages(mixed: bool, layers: int = 64):
    """Per layer {qkv}, {o}, {gate, up} (the same input), {down}; then the lm_head."""
    st = []
    for layer in range(layers):
        b = 5 * layer
        st += [[b], [b + 1], [b + 2, b + 3], [b + 4]]
    return st + ([[5 * layers]] if mixed else [])


def qwen3_8b_stack():
    """Qwen3-8B-shaped Q4_K stack ("Machine Learning on NVIDIA CMP", section "llama.cpp
    results", names Qwen3-8B Q4_K_M; every matrix here is Q4_K): 36 layers of
    {q 4096x4096, k and v 1024x4096 (8 KV heads of 128), o 4096x4096, gate and up
    12288x4096, down 4096x12288} plus the 151936x4096 lm_head."""
    layer = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096), (12288, 4096), (12288, 4096), (4096, 12288)]
    return [("q4_k", n, k) for _ in range(36) for (n, k) in layer] + [("q4_k", 151936, 4096)]


def qwen3_8b_stages():
    """Per layer {q, k, v}, {o}, {gate, up}, {down}; then the lm_head: 145 stages."""
    st = []
    for layer in range(36):
        b = 7 * layer
        st += [[b, b + 1, b + 2], [b + 3], [b + 4, b + 5], [b + 6]]
    return st + [[252]]


MLP_COPIES = 4   # 4 x 99 MB of weights per step: more than three times the 129 MB L2


def llama3_8b_mlp():
    """Llama-3-8B MLP (gate/up 14336x4096, down 4096x14336), rotated through
    MLP_COPIES distinct copies so that every step streams its weights from HBM."""
    return [("q4_0", 14336, 4096), ("q4_0", 14336, 4096), ("q4_0", 4096, 14336)] * MLP_COPIES


def llama3_8b_mlp_stages():
    """Per copy {gate, up} (the same input), then {down}."""
    return [st for c in range(MLP_COPIES) for st in ([3 * c, 3 * c + 1], [3 * c + 2])]


WORKLOADS = {
    "llama2_7b_q4_0_m1": dict(M=1, mats=llama2_7b_stack, stages=llama2_7b_stages,
                             desc="Llama-2-7B-shaped Q4_0 decode stack, M=1 (225 matrices + per-call Q8_1 quantize)"),
    "qwen3_8b_q4_k_m1": dict(M=1, mats=qwen3_8b_stack, stages=qwen3_8b_stages,
                             desc="Qwen3-8B-shaped Q4_K decode stack, M=1 (253 matrices + per-call Q8_1 quantize)"),
    "qwen3_8b_q4_k_m8": dict(M=8, mats=qwen3_8b_stack, stages=qwen3_8b_stages,
                             desc="Qwen3-8B-shaped Q4_K decode stack, M=8"),
    "nvfp4_27b_m1": dict(M=1, mats=lambda: dense_27b_stack(False), stages=lambda: dense_27b_stages(False),
                         desc="27B-class dense NVFP4 W4A16 stack, M=1"),
    "nvfp4_27b_m8": dict(M=8, mats=lambda: dense_27b_stack(False), stages=lambda: dense_27b_stages(False),
                         desc="27B-class dense NVFP4 W4A16 stack, M=8"),
    "mixed_27b_m1": dict(M=1, mats=lambda: dense_27b_stack(True), stages=lambda: dense_27b_stages(True),
                         desc="27B-class stack, FP8 attention every 4th layer + NVFP4 lm_head, M=1"),
    "mixed_27b_m8": dict(M=8, mats=lambda: dense_27b_stack(True), stages=lambda: dense_27b_stages(True),
                         desc="27B-class stack, FP8 attention every 4th layer + NVFP4 lm_head, M=8"),
    "nvfp4_27b_m16": dict(M=16, mats=lambda: dense_27b_stack(False), stages=lambda: dense_27b_stages(False),
                          desc="27B-class dense NVFP4 W4A16 stack, M=16"),
    "mixed_27b_m16": dict(M=16, mats=lambda: dense_27b_stack(True), stages=lambda: dense_27b_stages(True),
                          desc="27B-class stack, FP8 attention every 4th layer + NVFP4 lm_head, M=16"),
}
for _m in range(1, 9):
    WORKLOADS[f"llama3_8b_mlp_q4_0_m{_m}"] = dict(
        M=_m, mats=llama3_8b_mlp, stages=llama3_8b_mlp_stages,
        desc=f"Llama-3-8B MLP Q4_0 (gate/up 14336x4096, down 4096x14336), {MLP_COPIES} rotated copies, M={_m}")
# Single shapes, rotated through enough distinct copies (> 3x the 129 MB L2) that
# every call streams from HBM: the small single-matrix case and per-kernel profiling.
WORKLOADS["q4_0_4096sq_m1"] = dict(M=1, mats=lambda: [("q4_0", 4096, 4096)] * 48,
                                   desc="Q4_0 GEMV M=1, N=K=4096, 48 rotated copies")
WORKLOADS["q4_0_11008x4096_m1"] = dict(M=1, mats=lambda: [("q4_0", 11008, 4096)] * 16,
                                       desc="Q4_0 GEMV M=1, 11008x4096, 16 rotated copies")
WORKLOADS["q4_0_4096x11008_m1"] = dict(M=1, mats=lambda: [("q4_0", 4096, 11008)] * 16,
                                       desc="Q4_0 GEMV M=1, 4096x11008 (Llama-2-7B down), 16 rotated copies")
WORKLOADS["q4_0_14336x4096_m8"] = dict(M=8, mats=lambda: [("q4_0", 14336, 4096)] * 8,
                                       desc="Q4_0 M=8, 14336x4096 (Llama-3-8B gate), 8 rotated copies")
WORKLOADS["q4_k_12288x4096_m1"] = dict(M=1, mats=lambda: [("q4_k", 12288, 4096)] * 16,
                                       desc="Q4_K GEMV M=1, 12288x4096 (Qwen3-8B gate), 16 rotated copies")
for _m in (32, 96):
    WORKLOADS[f"fp8_7168x5120_m{_m}"] = dict(M=_m, mats=lambda: [("fp8", 7168, 5120)] * 12,
                                            desc=f"FP8 W8A16 7168x5120, M={_m} (one tcgen05 pass, K split over 2 CTAs), "
                                                 "12 rotated copies")
WORKLOADS["mixed_27b_m32"] = dict(M=32, mats=lambda: dense_27b_stack(True), stages=lambda: dense_27b_stages(True),
                                  desc="27B-class stack, FP8 attention every 4th layer + NVFP4 lm_head, M=32 "
                                       "(tcgen05, K split on the 5120/7168-row matrices)")
for _m in (1, 8, 16, 24, 32, 48, 64, 96):
    WORKLOADS[f"nvfp4_17408x5120_m{_m}"] = dict(M=_m, mats=lambda: [("nvfp4", 17408, 5120)] * 8,
                                               desc=f"NVFP4 W4A16 17408x5120, M={_m}, 8 rotated copies")
for _m in (1, 8, 16, 24, 48, 64):
    WORKLOADS[f"fp8_7168x5120_m{_m}"] = dict(M=_m, mats=lambda: [("fp8", 7168, 5120)] * 12,
                                            desc=f"FP8 W8A16 7168x5120, M={_m}, 12 rotated copies")
DEFAULT_WORKLOAD = "llama2_7b_q4_0_m1"


def weight_bytes(fmt, n, k):
    if fmt == "q4_0":
        return n * (k // 32) * Q4_0_BLOCK
    if fmt == "q4_k":
        return n * (k // 256) * Q4_K_BLOCK
    if fmt == "nvfp4":
        return n * k // 2 + n * k // 16
    return n * k + 4 * n   # fp8 + fp32 row scale


def act_bytes(fmt, M, k, fused=False):
    """Activation bytes a call reads: Q4_0 reads Q8_1 activations, or fp32 ones when
    the quantize is fused in (Q4_K likewise); NVFP4 and FP8 read fp16."""
    if fmt in ("q4_0", "q4_k"):
        return M * k * 4 if fused else M * (k // 32) * Q8_1_BLOCK
    return M * k * 2


def call_bytes(fmt, M, n, k, fused=False):
    """Algorithmic bytes of one call: weights + scales + activations + outputs."""
    return weight_bytes(fmt, n, k) + act_bytes(fmt, M, k, fused) + M * n * 4


# ----------------------------------------------------------------------------- host-side plumbing


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


class Dist:
    """Rank plumbing of a replica run: barrier and max over ranks (no-ops for one rank)."""

    def __init__(self, world: int, backend: str = "nccl", device=None):
        self.world = world
        self.device = device
        self.dist = None
        if world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                dist.init_process_group(backend, device_id=device)
            else:
                dist.init_process_group(backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v: float) -> float:
        if self.dist is None:
            return v
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def replica_rate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job rate of independent replicas: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / seconds_max


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"qmv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.fh.close()

    def summary(self):
        try:
            with open(self.path) as f:
                rows = [[c.strip() for c in ln.split(",")] for ln in f if ln.strip()]
            os.unlink(self.path)
        except OSError:
            rows = []
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


L2_BYTES = 129 * 10**6   # GB300 L2


def l2_note(weight_bytes: int) -> str:
    """How a workload keeps L2 from serving repeated steps: its weights outgrow it."""
    if weight_bytes <= L2_BYTES:
        raise ValueError(f"{weight_bytes} bytes of weights fit in L2: rotate more copies")
    return f"inputs larger than L2: every step streams {weight_bytes / 1e6:.0f} MB of weights (L2 129 MB)"


def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, bytes_per_launch: float):
    """DRAM bytes per launch of the bench's average launch, from a committed ncu
    capture of a few launches of the same kernel source (their DRAM bytes over their
    algorithmic bytes, times this launch's algorithmic bytes), or None when the source
    has changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel]
        if e.get("workload") != workload or e.get("source_sha") != source_digest(e["sources"]):
            return None
        return round(float(e["dram_bytes"]) / float(e["algorithmic_bytes"]) * bytes_per_launch)
    except (OSError, KeyError, ValueError, TypeError, ZeroDivisionError):
        return None


# ----------------------------------------------------------------------------- the GPU arm


class Stack:
    """Resident weights and per-call activation/output buffers of one workload."""

    def __init__(self, name: str, device, seed: int = 1234, fused: bool = True, grouped: bool = True, spec=None):
        """spec: dict(M, mats, stages) of a workload not in WORKLOADS (tests build
        reduced stacks of the same shapes through the same dispatch)."""
        import torch
        from gemm_qmv_quantize_gb300 import synth
        w = WORKLOADS[name] if spec is None else dict(M=spec["M"], mats=lambda: list(spec["mats"]),
                                                       stages=lambda: [list(st) for st in spec["stages"]])
        self.name, self.M, self.mats, self.device = name, w["M"], w["mats"](), device
        self.fused = fused
        # Dependent stages: matrices of a stage read the same input tensor and are
        # independent of each other; a grouped launch runs them together.
        deps = w["stages"]() if "stages" in w else [[i] for i in range(len(self.mats))]
        assert sorted(i for st in deps for i in st) == list(range(len(self.mats)))
        self.input_of = {i: j for j, st in enumerate(deps) for i in st}
        self.stages = deps if grouped else [[i] for i in range(len(self.mats))]
        M = self.M
        self.weights = []
        for i, (fmt, n, k) in enumerate(self.mats):
            s = seed * 100003 + i
            if fmt == "q4_0":
                self.weights.append((synth.q4_0_weights(n, k, s, device),))
            elif fmt == "q4_k":
                self.weights.append((synth.q4_k_weights(n, k, s, device),))
            elif fmt == "nvfp4":
                self.weights.append(synth.nvfp4_weights(n, k, s, device))
            else:
                self.weights.append(synth.fp8_weights(n, k, s, device))
        # activations (one per stage input) and outputs: views into two contiguous
        # buffers (one copy each way for e2e)
        first = [st[0] for st in deps]
        for st in deps:
            assert len({(self.mats[i][0], self.mats[i][2]) for i in st}) == 1, "a shared input has one format and K"
        x_is_f32 = [self.mats[i][0] in ("q4_0", "q4_k") for i in first]
        x_sizes = [M * self.mats[i][2] * (4 if f else 2) for i, f in zip(first, x_is_f32)]
        self.x_bytes = sum(x_sizes)
        self.x_buf = torch.empty(self.x_bytes, dtype=torch.uint8, device=device)
        inputs, off = [], 0
        for i, f, nbytes in zip(first, x_is_f32, x_sizes):
            dt = torch.float32 if f else torch.float16
            inputs.append(self.x_buf[off:off + nbytes].view(dt).view(M, self.mats[i][2]))
            off += nbytes
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        for x in inputs:
            x.copy_(torch.randn(x.shape, generator=g, device=device, dtype=torch.float32))
        self.xs = [inputs[self.input_of[i]] for i in range(len(self.mats))]
        self.y_elems = sum(M * n for _, n, _ in self.mats)
        self.y_buf = torch.empty(self.y_elems, dtype=torch.float32, device=device)
        self.ys, off = [], 0
        for _, n, _ in self.mats:
            self.ys.append(self.y_buf[off:off + M * n].view(M, n))
            off += M * n
        # Q8_1 activations of the two-call path: one buffer per stage input
        xq_in = [torch.empty((M, self.mats[i][2] // 32 * Q8_1_BLOCK), dtype=torch.uint8, device=device)
                 if self.mats[i][0] in ("q4_0", "q4_k") else None for i in first]
        self.xqs = [xq_in[self.input_of[i]] for i in range(len(self.mats))]
        self.bytes_per_step = sum(self.launch_bytes(st) for st in self.stages)
        self.weight_bytes = sum(weight_bytes(fmt, n, k) for fmt, n, k in self.mats)

    def run(self, events=None):
        """One step: every stage in stream order. events[j] = (start, end) around
        stage j's GEMV launch."""
        import gemm_qmv_quantize_gb300 as q
        for j, st in enumerate(self.stages):
            if len(st) > 1:
                fmt = self.mats[st[0]][0]
                if fmt in ("q4_0", "q4_k") and not self.fused:   # the stage's matrices share their input: quantize it once
                    q.qmv_quantize_q8_1(self.xs[st[0]], out=self.xqs[st[0]])
                if events is not None:
                    events[j][0].record()
                if fmt == "nvfp4":
                    q.qgemm_nvfp4_w4a16_group([self.weights[i][0] for i in st], [self.weights[i][1] for i in st],
                                              [self.weights[i][2] for i in st], self.xs[st[0]],
                                              [self.ys[i] for i in st])
                elif fmt == "fp8":
                    q.qgemm_fp8_w8a16_group([self.weights[i][0] for i in st], [self.weights[i][1] for i in st],
                                            self.xs[st[0]], [self.ys[i] for i in st])
                elif fmt == "q4_k" and self.fused:
                    q.qmv_q4_k_q8_1_fused_group([self.weights[i][0] for i in st], [self.xs[i] for i in st],
                                                [self.ys[i] for i in st])
                elif fmt == "q4_k":
                    q.qmv_q4_k_q8_1_group([self.weights[i][0] for i in st], [self.xqs[i] for i in st],
                                          self.mats[st[0]][2], [self.ys[i] for i in st])
                elif self.fused:
                    q.qmv_q4_0_q8_1_fused_group([self.weights[i][0] for i in st], [self.xs[i] for i in st],
                                                [self.ys[i] for i in st])
                else:
                    q.qmv_q4_0_q8_1_group([self.weights[i][0] for i in st], [self.xqs[i] for i in st],
                                          self.mats[st[0]][2], [self.ys[i] for i in st])
                if events is not None:
                    events[j][1].record()
                continue
            self._run_one(st[0], None if events is None else events[j])

    def _run_one(self, i, ev):
        import gemm_qmv_quantize_gb300 as q
        fmt, n, k = self.mats[i]
        x, y, wt = self.xs[i], self.ys[i], self.weights[i]
        if fmt in ("q4_0", "q4_k") and not self.fused:
            q.qmv_quantize_q8_1(x, out=self.xqs[i])
        if ev is not None:
            ev[0].record()
        if fmt == "q4_k" and self.fused:
            q.qmv_q4_k_q8_1_fused(wt[0], x, out=y)
        elif fmt == "q4_k":
            q.qmv_q4_k_q8_1(wt[0], self.xqs[i], k, out=y)
        elif fmt == "q4_0" and self.fused:
            q.qmv_q4_0_q8_1_fused(wt[0], x, out=y)
        elif fmt == "q4_0":
            q.qmv_q4_0_q8_1(wt[0], self.xqs[i], k, out=y)
        elif fmt == "nvfp4":
            q.qgemm_nvfp4_w4a16(wt[0], wt[1], wt[2], x, out=y)
        else:
            q.qgemm_fp8_w8a16(wt[0], wt[1], x, out=y)
        if ev is not None:
            ev[1].record()

    def launch_bytes(self, st):
        """Algorithmic bytes of one launch: weights, scales and outputs of its matrices,
        and each distinct input once."""
        b = sum(weight_bytes(fmt, n, k) + self.M * n * 4 for fmt, n, k in (self.mats[i] for i in st))
        for j in sorted({self.input_of[i] for i in st}):
            i = next(i for i in st if self.input_of[i] == j)
            b += act_bytes(self.mats[i][0], self.M, self.mats[i][2], self.fused)
        return b


def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()   # warm: attributes, lazy module loads
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def timed(replay, steps, barrier, sync):
    import torch
    barrier()
    sync()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        replay()
    end.record()
    sync()
    barrier()
    return start.elapsed_time(end) * 1e-3


def step_spread(replay, n):
    """Per-step device times of n more replays after the timed region (an event pair
    around each): median, p10 and p90 in ms. Reported beside the line's value, which
    comes from the timed region alone."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in ev:
        a.record()
        replay()
        b.record()
    torch.cuda.synchronize()
    ts = sorted(a.elapsed_time(b) for a, b in ev)

    def pick(f):
        return round(ts[min(n - 1, int(f * (n - 1) + 0.5))], 4)
    return {"n": n, "median_ms": pick(0.5), "p10_ms": pick(0.1), "p90_ms": pick(0.9)}


def q4_fused(args) -> bool:
    """Q4_0 path: the quantize fused into the MMVQ prologue at M = 1 (every CTA
    quantizes the row: cheaper than a launch); at M >= 2 the two-call path (one
    quantize per input, then MMVQ on Q8_1), unless a flag forces one."""
    if args.q4_path != "auto":
        return args.q4_path == "fused"
    return WORKLOADS[args.workload]["M"] == 1


def run_ours(args, rank, world, local_rank):
    import torch
    import gemm_qmv_quantize_gb300 as q
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = Dist(world, "nccl", dev)
    barrier, max_over_ranks = dist.barrier, dist.max

    stack = Stack(args.workload, dev, seed=1234 + rank, fused=q4_fused(args), grouped=not args.serial)
    stream = torch.cuda.Stream(device=dev)
    q.route_reset()
    q.set_launch_overlap(not args.no_overlap)
    with torch.cuda.stream(stream):
        line = _run_ours_on_stream(args, rank, world, local_rank, stack, stream, barrier, max_over_ranks)
    # secondary records: other workloads timed in the same run, each with its own roofline
    second = secondary_workloads(args)
    if second:
        del stack
        torch.cuda.empty_cache()
        line["secondary"] = []
        for wl in second:
            sargs = argparse.Namespace(**{**vars(args), "workload": wl, "steps": min(args.steps, 300)})
            try:
                st2 = Stack(wl, dev, seed=1234 + rank, fused=q4_fused(sargs), grouped=not args.serial)
                with torch.cuda.stream(stream):
                    rec = _run_ours_on_stream(sargs, rank, world, local_rank, st2, stream, barrier,
                                              max_over_ranks, secondary=True)
                del st2
            except Exception as exc:   # the main record stands; this one reports its failure
                rec = secondary_error(wl, exc)
            line["secondary"].append(rec)
            torch.cuda.empty_cache()
    dist.close()
    return line if rank == 0 else None


def secondary_error(workload, exc):
    """The record of a secondary workload that raised: its name and the error. The main
    record was measured before it and stands; this record carries no measurement and no
    parity verdict (a wrong result is still fatal: only a measured violation fails the
    run)."""
    return {"config": {"workload": workload}, "error": f"{type(exc).__name__}: {str(exc)[:300]}",
            "parity": {"ok": None, "error": "not measured"}}


def secondary_workloads(args):
    """Workloads timed after the main one in the same run: by default, beside the
    default Q4_0 stack, the 27B-class NVFP4 stack at M = 1 (the other M = 1 path whose
    HBM fraction is the target) and the mixed NVFP4/FP8 27B stack at M = 32 (the
    verification band on the tcgen05 kernel); none beside any other workload."""
    if args.secondary == "auto":
        return ["nvfp4_27b_m1", "mixed_27b_m32"] if args.workload == DEFAULT_WORKLOAD else []
    return [w for w in args.secondary.split(",") if w and w != "none"]


def _run_ours_on_stream(args, rank, world, local_rank, stack, stream, barrier, max_over_ranks, secondary=False):
    """The measured line of one workload: its timed region, roofline, clocks and, for
    the main record, e2e, parity and the CPU baseline (secondary records: parity only)."""
    import torch
    import gemm_qmv_quantize_gb300 as q
    q.route_reset()   # launches of one step, by the route census of an eager step
    stack.run()
    torch.cuda.synchronize()
    launches_per_step = sum(q.route_counts().values())
    if args.eager:
        replay = stack.run
    else:
        graph = capture(stack.run, stream)
        replay = graph.replay
    for _ in range(args.warmup):
        replay()
    torch.cuda.synchronize()
    launches0 = sum(q.route_counts().values())

    with ClockSampler(local_rank) as clocks:
        t_step_total = timed(replay, args.steps, barrier, torch.cuda.synchronize)
    t = max_over_ranks(t_step_total)
    ms_per_step = t / args.steps * 1e3
    step_s = t / args.steps
    gbs = replica_rate(stack.bytes_per_step, step_s, world) / 1e9
    kernels = launches_per_step * args.steps if not args.eager else sum(q.route_counts().values()) - launches0
    try:
        spread = step_spread(replay, max(1, min(args.steps, 200)))
    except RuntimeError as exc:   # a CUDA error here is reported in the line, not fatal to it
        spread = {"error": str(exc)[:200]}

    # dominant kernel: the GEMV of every call, timed per launch with event nodes in the graph
    roof = kernel_roofline(args, stack, stream, barrier, step_s=None if args.eager else step_s)

    # end to end through the public API with host buffers: pinned x in, y out, every step
    e2e = None if secondary else end_to_end(args, stack, replay, stream, barrier, max_over_ranks, world)

    err = q.error_flags(clear=True)
    peak, peak_kind = measured_peak()
    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(stack)[0],
        "dtype_detail": dtype_of(stack)[1], "data": "synthetic",
        "hbm_frac": round(gbs / world / peak, 4), "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
        "tok_per_s": round(stack.M * world / step_s, 1),
        "config": {"workload": stack.name, "desc": WORKLOADS[stack.name]["desc"], "M": stack.M,
                   "matrices": len(stack.mats), "weight_bytes": stack.weight_bytes,
                   "bytes_per_step": stack.bytes_per_step,
                   "l2": l2_note(stack.weight_bytes),
                   "launch": "eager" if args.eager else "cuda_graph", "launch_overlap": not args.no_overlap,
                   "q8_1_quantize": "fused into the MMVQ prologue" if stack.fused else
                   "two calls (quantize once per input, then MMVQ on Q8_1)",
                   "dependent_stages": len(stack.stages),
                   "schedule": ("one launch per matrix, each after the previous" if len(stack.stages) == len(stack.mats)
                                else "decode dependency structure: matrices reading the same input share a launch"),
                   "parallelism": f"replicas{world}"},
        "roofline": roof, "e2e": e2e, "step_ms": spread, "gpu_launches": int(kernels), "clocks": clocks.summary(),
        "device_error_flags": err,
    }
    if secondary:
        for key in ("metric", "unit", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "data", "e2e",
                    "hbm_peak_gbs", "hbm_peak_kind", "warmup"):
            line.pop(key, None)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["parity"] = sampled_parity(stack)
        if not secondary:
            line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds)
    return line


def dtype_of(stack):
    """(arithmetic type of the products, what the path computes in detail)."""
    fmts = {f for f, _, _ in stack.mats}
    if fmts <= {"q4_0", "q4_k"}:
        return "int8", "int8 x int8 block dots in int32 (dp4a / m16n8k32), fp32 scale and accumulate"
    return "fp16", "fp16 x fp16 tensor-core MMA (m16n8k16), fp32 accumulate; e2m1/e4m3 decode to fp16 is exact"


def kernel_roofline(args, stack, stream, barrier, step_s=None):
    """Roofline of the dominant kernel. Launches of a step overlap (programmatic
    dependent launch: each call's weight copies start while the previous call
    drains), so events bracketing every launch would serialise them and time a
    different program. When every launch of the step is the dominant kernel, its
    average launch duration is the timed region's device time over its launches
    (step_s / launches per step, from the CUDA events of the timed region); the
    bracketed per-launch figure is reported beside it as *_isolated. Otherwise
    (several kernels in the step) the bracketed figure is the achieved one."""
    import torch
    peak, peak_kind = measured_peak()
    n = len(stack.stages)
    try:
        events = [(torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n)]
        graph = capture(lambda: stack.run(events), stream)
        replay, how = graph.replay, "cuda_graph with event-record nodes"
    except TypeError:   # no external events: time eager launches instead
        events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]

        def replay():
            stack.run(events)
        how = "eager launches"
    for _ in range(max(1, args.warmup)):
        replay()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 200))
    total = [0.0] * n
    barrier()
    for _ in range(steps):
        replay()
        torch.cuda.synchronize()
        for j, (a, b) in enumerate(events):
            total[j] += a.elapsed_time(b) * 1e-3
    barrier()
    fmt_main = stack.mats[0][0]
    # the dominant kernel by the route census of one more (eager) step: the GEMV routes
    import gemm_qmv_quantize_gb300 as q
    q.route_reset()
    stack.run()
    torch.cuda.synchronize()
    routes = {k: v for k, v in q.route_counts().items() if v}
    gemv = {k: v for k, v in routes.items() if k.startswith(fmt_main)}
    kname = max(gemv, key=gemv.get) if gemv else fmt_main
    sel = [j for j, st in enumerate(stack.stages) if stack.mats[st[0]][0] == fmt_main]
    stage_bytes = [stack.launch_bytes(stack.stages[j]) for j in sel]
    bytes_per_launch = sum(stage_bytes) / len(sel)
    dur_iso = sum(total[j] for j in sel) / (len(sel) * steps)
    achieved_iso = bytes_per_launch / dur_iso / 1e9
    only = step_s is not None and set(routes) == {kname} and routes[kname] == len(stack.stages)
    if only:
        dur, achieved = step_s / routes[kname], bytes_per_launch / (step_s / routes[kname]) / 1e9
        timing = ("timed region: step time / launches per step (the only kernel in the step; launches "
                  "overlap); isolated: " + how)
    else:
        dur, achieved, timing = dur_iso, achieved_iso, how
    return {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": f"{peak_kind} (HBM copy bandwidth)", "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(kname, stack.name, bytes_per_launch), "bytes_per_launch": round(bytes_per_launch),
            "avg_launch_us": round(dur * 1e6, 3), "launches_timed": len(sel) * steps,
            "achieved_isolated": round(achieved_iso, 1), "frac_isolated": round(achieved_iso / peak, 4),
            "avg_launch_us_isolated": round(dur_iso * 1e6, 3), "timing": timing}


def end_to_end(args, stack, replay, stream, barrier, max_over_ranks, world):
    import torch
    x_host = torch.empty(stack.x_bytes, dtype=torch.uint8, pin_memory=True)
    x_host.copy_(stack.x_buf.cpu())
    y_host = torch.empty(stack.y_elems, dtype=torch.float32, pin_memory=True)
    steps = args.steps

    def one():   # all on the current stream (the bench stream)
        stack.x_buf.copy_(x_host, non_blocking=True)
        replay()
        y_host.copy_(stack.y_buf, non_blocking=True)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        one()
    end.record()
    torch.cuda.synchronize()
    barrier()
    t = max_over_ranks(max(start.elapsed_time(end) * 1e-3, 0.0))
    return {"value": round(stack.bytes_per_step * world / (t / steps) / 1e9, 1), "unit": "GB/s",
            "tok_per_s": round(stack.M * world / (t / steps), 1),
            "h2d_bytes_per_step": stack.x_bytes, "d2h_bytes_per_step": stack.y_elems * 4,
            "wall_s": round(time.perf_counter() - t0, 4)}


# ----------------------------------------------------------------------------- the oracle (CPU) arm


def host_threads() -> int:
    """Host cores this process may run on (the oracle's C calls release the GIL, so
    a thread per core runs the plain oracle in parallel over row blocks)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


class OracleSampler:
    """Times the CPU oracle on a bounded sample of a workload: for each distinct
    matrix shape, row blocks of one seeded matrix with the same per-call work (Q8_1
    quantize of the activation + the dot products), the time budget split across
    shapes in proportion to the stack's bytes, on `threads` host threads that take
    row blocks in turn. Inputs are generated once (untimed) and reused by every
    sample; the oracle itself is the plain, single-threaded C code."""

    BLOCK_ROWS = 64

    def __init__(self, workload: str, seed: int = 99):
        w = WORKLOADS[workload]
        self.M, mats = w["M"], w["mats"]()
        self.shapes = sorted(set(mats), key=mats.index)
        per_shape = {sh: sum(call_bytes(m[0], self.M, m[1], m[2]) for m in mats if m == sh) for sh in self.shapes}
        total = sum(per_shape.values())
        self.share = {sh: per_shape[sh] / total for sh in self.shapes}
        self.seed = seed
        self.cache = {}

    def _inputs(self, shape, rows):
        from gemm_qmv_quantize_gb300 import synth
        fmt, n, k = shape
        have = self.cache.get(shape)
        if have is None or have[0] < rows:
            r = min(n, max(rows, 2 * (have[0] if have else 0), 64))
            if fmt == "q4_0":
                w = (synth.q4_0_weights(r, k, self.seed, "cpu").numpy(),)
                x = synth.activations_f32(self.M, k, self.seed + 1, "cpu").numpy()
            elif fmt == "q4_k":
                w = (synth.q4_k_weights(r, k, self.seed, "cpu").numpy(),)
                x = synth.activations_f32(self.M, k, self.seed + 1, "cpu").numpy()
            elif fmt == "nvfp4":
                c, sc, g = synth.nvfp4_weights(r, k, self.seed, "cpu")
                w = (c.numpy(), sc.numpy(), g)
                x = synth.activations_f16(self.M, k, self.seed + 1, "cpu").numpy()
            else:
                wt, rs = synth.fp8_weights(r, k, self.seed, "cpu")
                w = (wt.numpy(), rs.numpy())
                x = synth.activations_f16(self.M, k, self.seed + 1, "cpu").numpy()
            self.cache[shape] = have = (r, w, x)
        return have

    def prepare(self):
        """Generate every shape's seeded inputs (untimed)."""
        for shape in self.shapes:
            self._inputs(shape, min(shape[1], 8192))

    def sample(self, budget_s: float, threads: int = 1):
        """(GB/s, info) of one bounded sample: `budget_s` seconds of wall time."""
        import itertools
        from concurrent.futures import ThreadPoolExecutor

        import numpy as np

        import oracle
        done_bytes, wall, rows_done = 0, 0.0, {}
        act = {sh: (self.M * (sh[2] // 32) * Q8_1_BLOCK if sh[0] in ("q4_0", "q4_k") else self.M * sh[2] * 2)
               for sh in self.shapes}
        for shape in self.shapes:
            fmt, n, k = shape
            key = f"{fmt} {n}x{k}"
            cap = min(n, 8192)   # rows of the seeded matrix, cycled through until the time share is used
            _, w, x = self._inputs(shape, cap)
            blocks = itertools.count()

            def one_call(off, r):
                if fmt == "q4_0":
                    oracle.q4_0_q8_1(np.ascontiguousarray(w[0][off:off + r]), oracle.quantize_q8_1(x), k)
                elif fmt == "q4_k":
                    oracle.q4_k_q8_1(np.ascontiguousarray(w[0][off:off + r]), oracle.quantize_q8_1(x), k)
                elif fmt == "nvfp4":
                    oracle.nvfp4_w4a16(np.ascontiguousarray(w[0][off:off + r]),
                                       np.ascontiguousarray(w[1][off:off + r]), w[2], x)
                else:
                    oracle.fp8_w8a16(np.ascontiguousarray(w[0][off:off + r]),
                                     np.ascontiguousarray(w[1][off:off + r]), x)

            def worker(deadline):
                b = r_done = 0
                while True:
                    off = (next(blocks) * self.BLOCK_ROWS) % cap
                    r = min(self.BLOCK_ROWS, cap - off)
                    one_call(off, r)
                    # the rows' weights and outputs, plus the activation once per call
                    b += weight_bytes(fmt, r, k) + self.M * r * 4 + act[shape]
                    r_done += r
                    if time.perf_counter() >= deadline:
                        return b, r_done

            t0 = time.perf_counter()
            deadline = t0 + budget_s * self.share[shape]
            with ThreadPoolExecutor(max_workers=threads) as ex:
                parts = list(ex.map(worker, [deadline] * threads))
            wall += time.perf_counter() - t0
            done_bytes += sum(p[0] for p in parts)
            rows_done[key] = sum(p[1] for p in parts)
        sample = (f"oracle (plain C, fp64) on {threads} host threads taking blocks of {self.BLOCK_ROWS} rows of one "
                  "seeded matrix per distinct shape (at most 8192 rows, cycled), wall time split by the stack's "
                  f"bytes per shape; rows processed per shape: {rows_done}")
        return done_bytes / wall / 1e9, {"bytes": done_bytes, "seconds": round(wall, 3), "sample": sample}


def cpu_baseline(workload: str, budget_s: float, threads: int | None = None):
    threads = threads or host_threads()
    sampler = OracleSampler(workload)
    sampler.prepare()
    gbs, info = sampler.sample(budget_s, threads)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": info["sample"],
            "seconds": info["seconds"]}


def sampled_parity(stack, rows: int = 8, seed: int = 7, threads: int | None = None):
    """Parity of the program that was timed, checked after the timed region (the
    cpu_baseline leg): for every matrix of the stack, `rows` sampled output rows (the
    first, the last and random ones) of the last step's y against the oracle on the
    same weights and activations, |y - y_ref| <= 1e-3 * sum_k |w x| + 1e-6."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import torch

    import oracle
    from gemm_qmv_quantize_gb300 import synth
    torch.cuda.synchronize()
    xs_host, jobs = {}, []
    for i, (fmt, n, k) in enumerate(stack.mats):
        ridx = synth.sample_rows(n, rows, seed + i).to(stack.device)
        j = stack.input_of[i]
        if j not in xs_host:
            xs_host[j] = stack.xs[i].cpu().numpy()
        w = tuple(t.index_select(0, ridx).cpu().numpy() if isinstance(t, torch.Tensor) else t
                  for t in stack.weights[i])
        jobs.append((fmt, k, w, j, stack.ys[i].index_select(1, ridx).cpu().numpy()))

    def check(job):
        fmt, k, w, j, y = job
        x = xs_host[j]
        if fmt == "q4_0":
            y_ref, bound = oracle.q4_0_q8_1(w[0], oracle.quantize_q8_1(x), k)
        elif fmt == "q4_k":
            y_ref, bound = oracle.q4_k_q8_1(w[0], oracle.quantize_q8_1(x), k)
        elif fmt == "nvfp4":
            y_ref, bound = oracle.nvfp4_w4a16(w[0], w[1], w[2], x)
        else:
            y_ref, bound = oracle.fp8_w8a16(w[0], w[1], x)
        if not np.all(np.isfinite(y)):
            return float("inf"), y.size
        return float(np.max(np.abs(y.astype(np.float64) - y_ref) / (1e-3 * bound + 1e-6))), y.size

    with ThreadPoolExecutor(max_workers=threads or host_threads()) as ex:
        res = list(ex.map(check, jobs))
    worst = max(r[0] for r in res)
    return {"matrices": len(jobs), "checked": int(sum(r[1] for r in res)), "rows_per_matrix": rows,
            "max_err_over_tol": round(worst, 4) if worst != float("inf") else "inf", "ok": bool(worst <= 1.0)}


def run_reference(args, rank, world):
    """The oracle as it stands, timed on this host's cores: each step is a bounded
    sample of the workload (--ref-seconds of wall time over the whole run); the line
    reports what was run -- the sample's bytes over its wall time, and the wall time
    of a sampled step -- and, under its own key, the time the whole stack would take
    at that rate."""
    if rank != 0:
        return None
    threads = host_threads()
    sampler = OracleSampler(args.workload)
    sampler.prepare()
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        sampler.sample(budget, threads)
    info, total_bytes = None, 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _, info = sampler.sample(budget, threads)
        total_bytes += info["bytes"]
    wall = time.perf_counter() - t0
    value = total_bytes / wall / 1e9
    w = WORKLOADS[args.workload]
    stack_bytes = sum(call_bytes(*m[:1], w["M"], *m[1:]) for m in w["mats"]())
    stack_s = stack_bytes / (value * 1e9)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / max(1, args.steps) * 1e3, 3),
        "step": f"one bounded sample of the workload: {round(total_bytes / max(1, args.steps))} bytes of "
                "weights, activations and outputs per step",
        "extrapolated_stack_ms": round(stack_s * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tok_per_s": round(w["M"] / stack_s, 4),
        "config": {"workload": args.workload, "desc": w["desc"], "M": w["M"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": info["sample"] if info else ""},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    p.add_argument("--eager", action="store_true", help="launch every call from Python (no CUDA graph)")
    p.add_argument("--q4-path", choices=["auto", "fused", "two_call"], default="auto",
                   help="Q4_0: quantize fused into the MMVQ prologue, or qmv_quantize_q8_1 then MMVQ on Q8_1; "
                        "auto = fused at M = 1, two calls from M = 2")
    p.add_argument("--serial", action="store_true",
                   help="one launch per matrix in stream order (no grouped launches of independent matrices)")
    p.add_argument("--no-overlap", action="store_true",
                   help="no programmatic dependent launch between consecutive calls")
    p.add_argument("--cpu-seconds", type=float, default=2.0,
                   help="wall-time budget of the cpu_baseline sample (on every host core)")
    p.add_argument("--ref-seconds", type=float, default=60.0,
                   help="oracle time budget of the whole --impl reference run")
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip the cpu_baseline leg (the oracle's timing and the sampled parity check)")
    p.add_argument("--secondary", default="auto",
                   help="comma-separated workloads timed after the main one in the same run ('none': no "
                        "secondary record; auto: the NVFP4 27B stack at M = 1 and the mixed 27B stack at "
                        "M = 32 beside the default workload)")
    return p.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if args.warmup < 3:
            print("warning: fewer than 3 warm-up steps", file=sys.stderr)
        line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
        bad = [r for r in [line] + line.get("secondary", []) if r.get("parity", {}).get("ok") is False]
        if bad:   # the timed program disagrees with the oracle: the line does not stand
            print("parity check failed: " + ", ".join(r["config"]["workload"] for r in bad), file=sys.stderr)
            sys.exit(1)


if __name__ == "__main__":
    main()

"""Host-side logic of bench.py on CPU: the replica plumbing across gloo ranks, the
workload tables, and the reference (oracle) arm under torchrun."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    d = bench.Dist(world, backend="gloo")
    d.barrier()
    local = 1.0 + rank            # rank 1 is the slow one
    t = d.max(local)
    out.put((rank, t, bench.replica_rate(100.0, t, world)))
    d.close()


def test_replicas_take_the_max_over_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]            # every rank sees the slowest time
    assert all(abs(r[2] - 100.0) < 1e-12 for r in res)  # 2 ranks x 100 units / 2 s


def test_single_rank_is_a_noop():
    d = bench.Dist(1)
    d.barrier()
    assert d.max(3.5) == 3.5
    d.close()


def test_workload_tables():
    mats = bench.llama2_7b_stack()
    assert len(mats) == 225
    assert sum(bench.weight_bytes(*m) for m in mats) == 3_716_481_024
    st = bench.llama2_7b_stages()
    assert len(st) == 129 and sorted(i for s in st for i in s) == list(range(225))
    mixed = bench.dense_27b_stack(True)
    assert sum(bench.weight_bytes(*m) for m in mixed) == 12_769_615_872
    dense = bench.dense_27b_stack(False)
    assert sum(bench.weight_bytes(*m) for m in dense) == 11_890_851_840
    assert sum(1 for f, _, _ in mixed if f == "fp8") == 32
    qwen = bench.qwen3_8b_stack()   # 36 x {q, o 4096^2; k, v 1024x4096; gate/up/down 12288x4096} + lm_head
    weights = 36 * (2 * 4096 ** 2 + 2 * 1024 * 4096 + 3 * 12288 * 4096) + 151936 * 4096
    assert sum(bench.weight_bytes(*m) for m in qwen) == weights * 144 // 256 == 4_257_054_720
    st = bench.qwen3_8b_stages()
    assert len(st) == 145 and sorted(i for s in st for i in s) == list(range(len(qwen)))
    mlp = bench.llama3_8b_mlp()     # one copy: 99,090,432 bytes
    assert sum(bench.weight_bytes(*m) for m in mlp) == 99_090_432 * bench.MLP_COPIES
    st = bench.llama3_8b_mlp_stages()
    assert sorted(i for s in st for i in s) == list(range(len(mlp)))


def test_every_workload_outgrows_l2():
    """Timing hygiene: no workload's weights fit in the 129 MB L2, so repeated steps
    stream from HBM (the single shapes and the MLP rotate copies, three L2s' worth)."""
    for name, w in bench.WORKLOADS.items():
        nbytes = sum(bench.weight_bytes(*m) for m in w["mats"]())
        assert nbytes > 2 * bench.L2_BYTES, name
        assert "129 MB" in bench.l2_note(nbytes)
    with pytest.raises(ValueError):
        bench.l2_note(99_090_432)


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--ref-seconds", "1.5",
           "--workload", "q4_0_4096sq_m1"]
    import time
    t0 = time.perf_counter()
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["dtype"] == "f64" and d["config"]["workload"] == "q4_0_4096sq_m1"
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cores"] == bench.host_threads()
    # the step time is one the run actually took (the extrapolation to the whole stack has its own key)
    assert d["steps"] * d["ms_per_step"] / 1e3 <= wall
    assert d["extrapolated_stack_ms"] > 0 and "bytes" in d["step"]


def test_step_spread_percentiles(monkeypatch):
    """The per-step spread reported beside the value: median, p10 and p90 of the
    event-pair times, here with a stand-in event clock (steps of 1..10 units)."""
    import torch
    clock = {"t": 0.0, "k": 0}

    class Ev:
        def __init__(self, enable_timing=True):
            self.v = None

        def record(self):
            clock["t"] += 1.0
            self.v = clock["t"]

        def elapsed_time(self, other):
            return other.v - self.v

    def replay():
        clock["k"] += 1
        clock["t"] += clock["k"] % 10

    monkeypatch.setattr(torch.cuda, "Event", Ev)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda: None)
    assert bench.step_spread(replay, 100) == {"n": 100, "median_ms": 6.0, "p10_ms": 2.0, "p90_ms": 9.0}
    assert bench.step_spread(replay, 1)["median_ms"] >= 1.0


def test_algorithmic_bytes_match_the_closed_forms():
    """The numerator of every GB/s figure: packed weights + scales + activations +
    outputs, per format, against the per-weight closed forms and the 4096 x 4096
    single-matrix and Llama-2-7B stack figures."""
    K = N = 4096
    assert bench.weight_bytes("q4_0", N, K) == N * K * 18 // 32 == 9_437_184
    assert bench.weight_bytes("q4_k", N, K) == N * K * 144 // 256
    assert bench.weight_bytes("nvfp4", N, K) == N * K // 2 + N * K // 16      # 0.5625 B per weight
    assert bench.weight_bytes("fp8", N, K) == N * K + 4 * N                    # + fp32 row scale
    assert bench.call_bytes("q4_0", 1, N, K) == 9_437_184 + 4_608 + 16_384     # Q8_1 in, fp32 out
    assert bench.call_bytes("q4_0", 1, N, K, fused=True) == 9_437_184 + 16_384 + 16_384   # fp32 in
    assert bench.call_bytes("nvfp4", 8, N, K) == bench.weight_bytes("nvfp4", N, K) + 8 * K * 2 + 8 * N * 4
    mats = bench.llama2_7b_stack()
    assert sum(4 * n for _, n, _ in mats) == 5_567_488                         # outputs of one token
    assert sum((k // 32) * 36 for _, _, k in mats) == 1_285_632                # one Q8_1 row per matmul


def test_secondary_records_beside_the_default_workload():
    """The default line also times the 27B NVFP4 stack at M = 1 and the mixed 27B stack
    at M = 32 (the tcgen05 band); other workloads carry no secondary record unless asked."""
    import bench
    args = bench.parse_args([])
    assert bench.secondary_workloads(args) == ["nvfp4_27b_m1", "mixed_27b_m32"]
    assert all(w in bench.WORKLOADS for w in bench.secondary_workloads(args))
    assert bench.secondary_workloads(bench.parse_args(["--workload", "nvfp4_27b_m8"])) == []
    assert bench.secondary_workloads(bench.parse_args(["--secondary", "none"])) == []
    assert bench.secondary_workloads(bench.parse_args(["--secondary", "mixed_27b_m16"])) == ["mixed_27b_m16"]


def test_secondary_error_record_keeps_the_line():
    """A secondary workload that raises leaves an error record beside the main record,
    with no parity verdict (only a measured violation fails the run)."""
    import bench
    rec = bench.secondary_error("mixed_27b_m32", RuntimeError("CUDA error: out of memory"))
    assert rec["config"]["workload"] == "mixed_27b_m32"
    assert rec["error"].startswith("RuntimeError: CUDA error")
    assert rec["parity"]["ok"] is None and "value" not in rec

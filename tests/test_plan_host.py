"""Host-side dispatch (the per-(M, N, K) launch heuristic) on the CPU: the Q4_0 /
Q4_K streaming-kernel plans for a GB300 (152 SMs, 227 KB of shared memory per
block), through qmv_debug_plan_q4, which runs the same planner as every call
without touching a GPU.

- The plans of the Llama-2-7B-shaped stack, the Llama-3-8B MLP sweep and the
  Qwen3-8B-shaped Q4_K stack: register-resident activation records at M = 1 with
  rows of 16 units, at M = 2..3 for Q4_0; lane pairs at M = 4; shared-memory
  records where a lane's unit changes from chunk to chunk (K = 11008, 14336).
- The generic kernel where the streaming one cannot run: K not a multiple of 256,
  weights not 16-byte aligned, activations too large to stage.
- Invariants over a sweep of shapes: shared memory within the device's limit, one
  CTA per SM at most, register records only where a lane keeps its unit.
The tensor-core kernel's plan (M >= 5) queries the device's occupancy, so the sweep
moves its threshold past M = 8 to see the streaming plans at every M.
"""
import pytest

from gemm_qmv_quantize_gb300 import _binding
from gemm_qmv_quantize_gb300._binding import GB300_DEVICE, QmvError, qmv_debug_plan_q4 as plan

STREAM = {False: "q4_0_stream_dp4a", True: "q4_k_stream_dp4a"}


SPARE = GB300_DEVICE["sm_count"] // 12   # SMs the streaming grid leaves free (12 of 152)


@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 4096), (22016, 4096), (32000, 4096)])
def test_llama2_7b_rows_of_16_units_keep_records_in_registers(N, K):
    p = plan(1, N, K)
    assert p == dict(route="q4_0_stream_dp4a", warps=16, slots=2, grid=152 - SPARE, smem_bytes=p["smem_bytes"],
                     act_regs=1, pair=0, chunk_units=32)


def test_stream_grid_leaves_spare_sms(monkeypatch):
    """In a chain of calls the next call's last CTA lands on the SM that finished last;
    the grid leaves one SM in twelve free so that no straggler of the previous call
    takes a CTA of the next (measured: 3935 -> 4245 GB/s on the Llama-2-7B stack)."""
    assert plan(1, 4096, 11008)["grid"] == 140
    assert plan(1, 16 * 9 + 1, 4096)["grid"] == 10          # small N: fewer CTAs than SMs anyway
    monkeypatch.setenv("QMV_Q4_SPARE_SMS", "0")
    assert plan(1, 4096, 11008)["grid"] == 152
    small = dict(sm_count=8, smem_optin=101376, smem_per_sm=102400)
    monkeypatch.delenv("QMV_Q4_SPARE_SMS")
    assert plan(1, 4096, 4096, **small)["grid"] == 8        # 8 // 12 = 0 spare SMs


def test_down_projection_reads_records_from_shared_memory():
    p = plan(1, 4096, 11008)    # 43 units per row: a lane's unit changes from chunk to chunk
    assert p["route"] == "q4_0_stream_dp4a" and p["act_regs"] == 0 and p["warps"] == 16


@pytest.mark.parametrize("M,act_regs,pair,warps,slots", [(1, 1, 0, 16, 2), (2, 1, 0, 8, 4), (3, 1, 0, 8, 4),
                                                         (4, 0, 1, 8, 2)])
def test_llama3_8b_gate_up_plans(M, act_regs, pair, warps, slots):
    p = plan(M, 2 * 14336, 4096)
    assert (p["route"], p["act_regs"], p["pair"], p["warps"], p["slots"]) == \
        ("q4_0_stream_dp4a", act_regs, pair, warps, slots)


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_llama3_8b_down_plans(M):
    p = plan(M, 4096, 14336)    # 56 units per row
    assert p["route"] == "q4_0_stream_dp4a" and p["act_regs"] == 0 and p["pair"] == 0


def test_q4_k_registers_at_m1_only():
    assert plan(1, 12288, 4096, q4k=True)["act_regs"] == 1
    p = plan(2, 12288, 4096, q4k=True)
    assert p["route"] == "q4_k_stream_dp4a" and p["act_regs"] == 0 and p["pair"] == 0 and p["warps"] == 16


def test_generic_kernel_where_the_stream_cannot_run():
    assert plan(1, 100, 4128)["route"] == "q4_0_generic"                    # K % 256 != 0
    assert plan(1, 4096, 4096, w_align16=False)["route"] == "q4_0_generic"  # rows not 16-byte aligned
    assert plan(4, 40, 65536)["route"] == "q4_0_generic"                    # 4 x 256 records do not fit
    p = plan(1, 40, 65536)                                                  # one row of records does
    assert p["route"] == "q4_0_stream_dp4a" and p["smem_bytes"] <= GB300_DEVICE["smem_optin"]


def test_small_n_launches_only_the_ctas_it_needs():
    assert plan(1, 5, 4096)["grid"] == 1
    assert plan(1, 16 * 9 + 1, 4096)["grid"] == 10


def test_shape_and_pointer_validation():
    lib = _binding.lib()
    out = (_binding.ctypes.c_int64 * 8)()
    dev = (152, 232448, 233472)
    assert lib.qmv_debug_plan_q4(0, 1, 64, 4096, 1, 1, *dev, None) == -1        # QMV_ERR_NULL
    for bad in [(0, 9, 64, 4096, 1, 1), (0, 1, 64, 4100, 1, 1), (1, 1, 64, 4128, 1, 1), (0, 1, 64, 4096, 9, 1),
                (0, 1, 2, 4096, 3, 1), (0, 0, 64, 4096, 1, 1)]:
        assert lib.qmv_debug_plan_q4(*bad, *dev, out) == -2, bad                # QMV_ERR_SHAPE
    assert lib.qmv_debug_plan_q4(0, 1, 64, 4096, 1, 1, 0, 232448, 233472, out) == -2
    with pytest.raises(QmvError, match="QMV_ERR_SHAPE"):
        plan(1, 64, 4096, n_inputs=0)


def _sweep():
    for q4k in (False, True):
        for M in range(1, 9):
            for K in (256, 512, 1024, 4096, 4128, 11008, 12288, 14336, 16384, 65536):
                if q4k and K % 256:
                    continue
                for N in (1, 37, 4096, 151936):
                    for n_inputs in (1, 3):
                        if N >= n_inputs:
                            yield q4k, M, N, K, n_inputs


def test_plan_invariants_over_shapes(monkeypatch):
    monkeypatch.setenv("QMV_Q4_MMA_MIN_M", "9")
    monkeypatch.setenv("QMV_Q4K_MMA_MIN_M", "9")
    seen = set()
    for q4k, M, N, K, n_inputs in _sweep():
        p = plan(M, N, K, q4k=q4k, n_inputs=n_inputs)
        seen.add(p["route"])
        if p["route"] != STREAM[q4k]:
            # no streaming plan; for Q4_K that means no kernel at all (the call refuses the shape)
            assert p["route"] == "q4_0_generic", (q4k, M, N, K)
            records = (M * n_inputs * (K // 256) * 336 + 127) // 128 * 128
            assert K % 256 or records + 2 * 32 * 144 + 16 > GB300_DEVICE["smem_optin"]   # + one warp's ring
            continue
        U = K // 256
        assert 0 < p["smem_bytes"] <= GB300_DEVICE["smem_optin"], (q4k, M, N, K)
        assert 1 <= p["grid"] <= GB300_DEVICE["sm_count"]
        assert p["warps"] * 32 <= (512 if M < 3 or p["act_regs"] else 256)
        assert p["chunk_units"] == 32 and 1 <= p["slots"] <= 8
        assert p["grid"] * p["warps"] >= min(N, (GB300_DEVICE["sm_count"] - SPARE) * p["warps"]) or N < p["warps"]
        if p["act_regs"]:
            assert 32 % U == 0 and (M == 1 or (not q4k and M <= 3))
        if p["pair"]:
            assert M == 4 and U == 16 and not q4k and not p["act_regs"]
    assert seen == {"q4_0_stream_dp4a", "q4_0_generic", "q4_k_stream_dp4a"}


def test_smaller_device_degrades_to_fewer_warps_or_the_generic_kernel():
    small = dict(sm_count=8, smem_optin=101376, smem_per_sm=102400)   # 99 KB of shared memory per block
    p = plan(1, 4096, 4096, **small)
    assert p["route"] == "q4_0_stream_dp4a" and p["smem_bytes"] <= small["smem_optin"] and p["grid"] <= 8
    assert p["warps"] < 16
    assert plan(1, 64, 65536, **small)["warps"] == 1                  # 86 KB of records: one warp's ring left
    assert plan(2, 64, 65536, **small)["route"] == "q4_0_generic"     # 172 KB: no streaming plan

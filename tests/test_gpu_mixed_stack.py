"""GPU: the per-region dispatch of the mixed NVFP4 / FP8 27B-class stack, run as the
benchmark runs it, against the oracle, with the route census checked for fallbacks.

"v100-skinny README", section "Native mixed-precision checkpoint path": every weight
region goes to the kernel of its format -- FP8 attention regions to the FP8 kernel,
NVFP4 regions to the NVFP4 kernel, at M = 1..8, 9..16 (two row tiles per weight pass)
and 17..96 (chunks of <= 16 rows) -- and the census of the routes taken is checked
for fallbacks. The stack here is the benchmark's mixed stack cut to its first four
layers (layer 3 carries the FP8 qkv and o projections) plus the 151936 x 5120 NVFP4
lm_head, all at their real shapes, dispatched by the same code (bench.Stack.run, with
programmatic dependent launch on, as the benchmark runs it). Every matrix's sampled
rows (first, last, random) are compared with the oracle within
|y - y_ref| <= 1e-3 * sum|w x| + 1e-6, and the census must show exactly one launch
(per chunk of 16 rows) of the FP8 kernel per FP8 region and of the NVFP4 kernel per
NVFP4 stage, and no generic kernel: every stage on the kernel the planner chooses
for it (mma.sync up to 8 rows; from 9 rows the tcgen05 kernel for matrices of few
128-row tiles, the 5120-row ones here; from 17 rows the tcgen05 kernel everywhere).
"""
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu
LAYERS = 4


@pytest.fixture(scope="module")
def q():
    from gemm_qmv_quantize_gb300 import build
    build.build()
    import gemm_qmv_quantize_gb300 as q
    before = q.get_launch_overlap()
    q.set_launch_overlap(True)
    yield q
    q.set_launch_overlap(before)


@pytest.mark.parametrize("M", [1, 8, 16, 32, 48])
def test_mixed_stack_regions_dispatch_and_match_the_oracle(q, M):
    spec = dict(M=M, mats=bench.dense_27b_stack(True, LAYERS), stages=bench.dense_27b_stages(True, LAYERS))
    stack = bench.Stack(f"mixed_27b_{LAYERS}layers_m{M}", torch.device("cuda"), seed=77 + M, spec=spec)
    assert sum(1 for f, _, _ in stack.mats if f == "fp8") == 2 and stack.mats[-1] == ("nvfp4", 151936, 5120)
    q.error_flags(clear=True)
    q.route_reset()
    stack.run()
    torch.cuda.synchronize()
    counts = {k: v for k, v in q.route_counts().items() if v}
    fp8_stages = sum(1 for st in stack.stages if stack.mats[st[0]][0] == "fp8")
    nvfp4_stages = len(stack.stages) - fp8_stages
    assert (fp8_stages, nvfp4_stages) == (2, 4 * LAYERS + 1 - 2)
    # the kernel of every stage as the planner chooses it (its host logic is pinned on the
    # CPU): launches per stage = its chunks of <= 16 rows on the mma.sync route, 1 otherwise
    want = {}
    for st in stack.stages:
        fmt, _, K = stack.mats[st[0]]
        plan = q.qmv_debug_plan_wq(M, K, [stack.mats[i][1] for i in st], fp4=fmt == "nvfp4")
        want[plan["route"]] = want.get(plan["route"], 0) + plan["chunks"]
    assert sum(want.values()) >= len(stack.stages)
    if M >= 17:
        assert set(want) == {"nvfp4_tcgen05", "fp8_tcgen05"}
    if M <= 8:
        assert set(want) == {"nvfp4_mma_m16n8k16", "fp8_mma_m16n8k16"}
    assert counts == want, counts
    assert not any(k.endswith("generic") for k in counts)
    par = bench.sampled_parity(stack, rows=8)
    print(f"M={M}: {par}")
    assert par["matrices"] == len(stack.mats) and par["checked"] == 8 * M * len(stack.mats)
    assert par["ok"], par
    assert q.error_flags() == 0

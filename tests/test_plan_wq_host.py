"""Host-side dispatch of the NVFP4 / FP8 tensor-core kernel on the CPU, through
qmv_debug_plan_wq: the same candidate scoring as every launch, with the CTAs per
SM taken from an occupancy model (registers, shared memory, resident warps) instead
of the device, so no GPU is needed.

- Choices the design notes measured and kept: three 8-warp CTAs per SM at M = 1
  (the 5120 x 17408 down projection and the lm_head), 16 warps sharing one staged
  copy of the activations at M = 8 with K = 5120, two 8-row activation tiles in one
  weight pass at M = 9..16, then one pass on the tcgen05 kernel (from 17 rows; from 9
  for launches of at most a third of the SMs' worth of tiles) or balanced chunks of
  <= 16 rows ("v100-skinny README", "Native
  mixed-precision checkpoint path": the qpn8 / qpn8-mt2 / qpn8-chunked routes), the
  generic kernel for unaligned data or K off the step.
- Invariants over a sweep of shapes, M and register limits: shared memory within the
  device's opt-in limit and the SM, the grid = min(tiles, SMs x CTAs per SM), every
  warp the same number of steps per round, passes dividing the steps, the staged
  activation slice within its budget.
"""
import math

import pytest

from gemm_qmv_quantize_gb300._binding import GB300_DEVICE, QmvError, qmv_debug_plan_wq as plan

MMA = {True: "nvfp4_mma_m16n8k16", False: "fp8_mma_m16n8k16"}
UMMA = {True: "nvfp4_tcgen05", False: "fp8_tcgen05"}
UMMA_MIN_M = {True: 17, False: 17}   # launches of many tiles (17408 rows: 136)
GENERIC = {True: "nvfp4_generic", False: "fp8_generic"}
SHAPES_27B = [(7168, 5120), (5120, 5120), (17408, 5120), (5120, 17408), (151936, 5120)]


def _step_k(fp4):
    return 256 if fp4 else 128


@pytest.mark.parametrize("N,K", [(5120, 17408), (151936, 5120), (7168, 5120)])
def test_m1_three_8_warp_ctas_per_sm(N, K):
    p = plan(1, K, N)
    assert (p["route"], p["warps"], p["ctas_per_sm"]) == (MMA[True], 8, 3)
    assert p["grid"] == min(math.ceil(N / 16), 152 * 3)


@pytest.mark.parametrize("fp4", [True, False])
def test_m8_k5120_sixteen_warps_share_the_staged_activations(fp4):
    p = plan(8, 5120, 17408, fp4=fp4)
    assert (p["warps"], p["staged"], p["ctas_per_sm"], p["passes"]) == (16, 1, 1, 1)


@pytest.mark.parametrize("M", range(9, 17))
@pytest.mark.parametrize("fp4", [True, False])
def test_m9_to_16_one_weight_pass(M, fp4):
    p = plan(M, 5120, 7168, fp4=fp4)
    assert (p["route"], p["chunks"], p["chunk_rows"]) == (MMA[fp4], 1, M)


@pytest.mark.parametrize("M", [17, 24, 32, 33, 48, 64, 95, 96])
def test_chunked_band(M, monkeypatch):
    """Without the tcgen05 kernel (QMV_WQ_UMMA_MIN_M=0) rows above 16 go in balanced chunks."""
    monkeypatch.setenv("QMV_WQ_UMMA_MIN_M", "0")
    p = plan(M, 5120, 7168, fp4=False)
    chunks = math.ceil(M / 16)
    assert (p["route"], p["chunks"], p["chunk_rows"]) == (MMA[False], chunks, math.ceil(M / chunks))
    assert p["chunk_rows"] <= 16


@pytest.mark.parametrize("fp4", [True, False])
@pytest.mark.parametrize("M", [16, 17, 24, 32, 33, 48, 64, 80, 96])
def test_tcgen05_band(fp4, M):
    """From 17 rows one pass on the tcgen05 kernel: 128-row tiles; T
    issuing threads with an accumulator of 16 ceil(M / 16) columns each and Q >= max(T, 2)
    64-k A buffers of 32 columns (a multiple of 3 and of T: three decode groups take
    turns on the buffers, and thread t's buffers were last used by its own quarters),
    all within the 512 columns of tensor memory (the A
    buffers from the first 32-aligned column after the accumulators); R >= T activation
    slices; at least 3 weight stages; shared memory within the device's limit."""
    N, K = 17408, 5120
    p = plan(M, K, N, fp4=fp4)
    if M < UMMA_MIN_M[fp4]:
        assert p["route"] == MMA[fp4]
        return
    n_pad = 16 * math.ceil(M / 16)
    assert (p["route"], p["chunks"], p["chunk_rows"]) == (UMMA[fp4], 1, M)
    T, Q, R = p["warps"], p["a_bufs"], p["b_bufs"]
    # Q a multiple of the 3 decode groups and of T: the buffer an issuing thread waits
    # on was last used by one of its own earlier quarters
    assert 1 <= T <= 8 and Q >= max(T, 2) and Q % (3 // math.gcd(3, T) * T) == 0 and R >= max(T, 2)
    assert 32 * math.ceil(T * n_pad / 32) + 32 * Q <= 512
    assert Q >= min(6, (512 - 32 * math.ceil(T * n_pad / 32)) // 32)   # room for the decode to run ahead
    assert 3 <= p["slots"] <= 12 and p["smem_bytes"] <= GB300_DEVICE["smem_optin"]
    assert p["grid"] == min(math.ceil(N / 128), GB300_DEVICE["sm_count"])


def test_generic_routes():
    assert plan(3, 5120 + 16, 7168)["route"] == GENERIC[True]          # K off the 256-k step
    assert plan(3, 5120, 7168, aligned16=False)["route"] == GENERIC[True]
    p = plan(20, 5000, 7168, fp4=False)                                  # K off the 128-k step
    assert (p["route"], p["chunks"], p["chunk_rows"]) == (GENERIC[False], 3, 8)


def test_group_tiles_add_up():
    one = plan(1, 5120, 17408)
    two = plan(1, 5120, [17408, 17408])
    assert two["grid"] == min(2 * 17408 // 16, 152 * two["ctas_per_sm"])
    assert one["route"] == two["route"] == MMA[True]


def test_rejects_bad_arguments():
    with pytest.raises(QmvError):
        plan(0, 5120, 7168)
    with pytest.raises(QmvError):
        plan(97, 5120, 7168)
    with pytest.raises(QmvError):
        plan(1, 5120, [7168] * 9)
    with pytest.raises(QmvError):
        plan(1, 5120 + 16, [7168, 7168])   # a group needs the tensor-core kernel's K step
    with pytest.raises(QmvError):
        plan(40, 5120 + 16, [7168, 7168])
    with pytest.raises(QmvError):
        plan(1, 5120, 7168, ctas_by_regs=(0, 1, 1))


@pytest.mark.parametrize("fp4", [True, False])
@pytest.mark.parametrize("regs", [(3, 2, 1), (4, 2, 2), (1, 1, 1)])
def test_invariants_over_a_sweep(fp4, regs):
    dev = GB300_DEVICE
    for N, K in SHAPES_27B + [(16 * 37 + 5, 5120), (4096, 4096), (1, 256), (40, 768), (100, 65536)]:
        if K % _step_k(fp4):
            continue
        for M in (1, 2, 3, 5, 8, 9, 12, 16, 17, 40, 96):
            p = plan(M, K, N, fp4=fp4, ctas_by_regs=regs)
            rows = p["chunk_rows"]
            few = math.ceil(N / 128) * 3 <= dev["sm_count"]
            if M >= UMMA_MIN_M[fp4] or (few and M >= 9):
                assert p["route"] == UMMA[fp4] and rows == M
                continue
            assert p["route"] == MMA[fp4]
            assert 1 <= rows <= 16 and p["chunks"] == (math.ceil(M / 16) if M > 16 else 1)
            assert p["warps"] in (8, 16) and 2 <= p["slots"] <= 4
            assert 1 <= p["ctas_per_sm"] <= min(4, regs[2 if p["warps"] == 16 else (1 if rows > 8 else 0)])
            assert p["smem_bytes"] <= dev["smem_optin"]
            assert p["ctas_per_sm"] * (p["smem_bytes"] + 1024) <= dev["smem_per_sm"]
            assert p["ctas_per_sm"] * p["warps"] <= 64
            tiles = math.ceil(N / 16)
            assert p["grid"] == min(tiles, dev["sm_count"] * p["ctas_per_sm"])
            steps = K // _step_k(fp4)
            assert steps % p["passes"] == 0
            per_pass = steps // p["passes"]
            # every warp gets the same number of steps in a full round
            assert (p["tiles_per_round"] * per_pass) % p["warps"] == 0
            if p["staged"]:
                assert rows * (2 * K // p["passes"] + 16) <= 200 * 1024
            else:
                assert p["passes"] == 1


@pytest.mark.parametrize("fp4,N,K,want", [
    (True, 17408, 5120, 1), (False, 17408, 5120, 1),   # 136 tiles: no split
    (True, 7168, 5120, 2), (False, 7168, 5120, 2),     # 56 tiles: 152 // 56
    (True, 5120, 5120, 3), (False, 5120, 17408, 3),    # 40 tiles: 152 // 40
    (True, 2048, 4096, 4), (False, 2048, 4096, 4),     # 16 tiles: capped at 4
    (True, 151936, 5120, 1),                           # lm_head: persistent grid
    (True, 128, 256, 1), (False, 128, 256, 2),         # one tile: capped by the K steps (1 / 2)
    (True, 256, 768, 3), (False, 256, 384, 3)])
def test_tcgen05_split_k(fp4, N, K, want):
    """Split K when the tiles leave half the SMs idle: floor(152 / tiles) CTAs per tile,
    at most 4 and at most the K steps (NVFP4 steps of 256 k, FP8 of 128 k); the grid
    is tiles x splits, never more than the SMs."""
    tiles = math.ceil(N / 128)
    p = plan(96, K, N, fp4=fp4)
    assert p["k_splits"] == want
    assert p["grid"] == (tiles * want if want > 1 else min(tiles, GB300_DEVICE["sm_count"]))
    assert p["grid"] <= GB300_DEVICE["sm_count"]


@pytest.mark.parametrize("fp4", [True, False])
@pytest.mark.parametrize("N,few", [(301, True), (5120, True), (128 * 50, True), (128 * 51, False),
                                   (7168, False), (17408, False)])
@pytest.mark.parametrize("M", [8, 9, 16, 17])
def test_tcgen05_few_tiles_band(fp4, N, few, M):
    """From 9 rows the tcgen05 kernel takes launches of at most a third of the SMs' worth
    of 128-row tiles (50 of 152: K split over 3+ CTAs of a cluster), from 17 rows every
    launch; below that the mma.sync kernel in one pass."""
    p = plan(M, 5120, N, fp4=fp4)
    umma = M >= 17 or (few and M >= 9)
    assert p["route"] == (UMMA if umma else MMA)[fp4]
    if umma and few:
        assert p["k_splits"] >= 3


def test_tcgen05_thresholds_follow_the_environment(monkeypatch):
    """QMV_WQ_UMMA_MIN_M = 0 keeps the tcgen05 kernel off everywhere; 1 takes it for every
    M; QMV_WQ_UMMA_FEW_TILES_MIN_M moves the few-tile threshold alone."""
    monkeypatch.setenv("QMV_WQ_UMMA_MIN_M", "0")
    assert plan(16, 5120, 5120)["route"] == MMA[True] and plan(96, 5120, 301)["route"] == MMA[True]
    monkeypatch.setenv("QMV_WQ_UMMA_MIN_M", "1")
    assert plan(1, 5120, 17408)["route"] == UMMA[True] and plan(1, 5120, 301)["route"] == UMMA[True]
    monkeypatch.delenv("QMV_WQ_UMMA_MIN_M")
    monkeypatch.setenv("QMV_WQ_UMMA_FEW_TILES_MIN_M", "17")
    assert plan(16, 5120, 5120)["route"] == MMA[True] and plan(17, 5120, 5120)["route"] == UMMA[True]

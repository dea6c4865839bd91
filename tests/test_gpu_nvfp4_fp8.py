"""GPU parity: NVFP4 W4A16 and FP8 W8A16 skinny GEMM through the C ABI vs the CPU oracle.

fp32 outputs within |y - y_ref| <= 1e-3 * sum|w*x| + 1e-6 on: several tiles with
a ragged tail at M = 1..16 (rows 9..16 as a second activation tile of the same
weight pass) and chunked M up to 96; the full-size matrices of the 27B-class dense stack
and its 151936-row lm_head (sampled rows); fp16 activation outliers up to
6e4 (the overflow case of "v100-skinny README", section "How QPN works");
zero scales; K that is not a multiple of the streaming step (generic kernel).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_ABS, TOL_REL, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def q():
    from gemm_qmv_quantize_gb300 import build
    build.build()
    import gemm_qmv_quantize_gb300 as q
    return q


@pytest.fixture(autouse=True)
def mma_below_17_rows(monkeypatch):
    """These tests are about the mma.sync kernel: launches of few tiles keep it up to 16
    rows (by default they take the tcgen05 kernel from 9 rows; see
    test_default_dispatch below)."""
    monkeypatch.setenv("QMV_WQ_UMMA_FEW_TILES_MIN_M", "17")


def _synth():
    from gemm_qmv_quantize_gb300 import synth
    return synth


def _nvfp4(q, M, N, K, seed, outliers=0, rows=None, g=None):
    synth = _synth()
    codes, scales, g0 = synth.nvfp4_weights(N, K, seed=seed, device=DEV)
    g = g0 if g is None else g
    x = synth.activations_f16(M, K, seed=seed + 1, device=DEV, outliers=outliers)
    y = q.qgemm_nvfp4_w4a16(codes, scales, g, x).cpu().numpy()
    rows = np.arange(N) if rows is None else rows
    y_ref, bound = oracle.nvfp4_w4a16(codes.cpu().numpy()[rows], scales.cpu().numpy()[rows], g, x.cpu().numpy())
    assert_close(f"nvfp4 M={M} N={N} K={K}", y[:, rows], y_ref, bound)
    return y


def _fp8(q, M, N, K, seed, outliers=0, rows=None):
    synth = _synth()
    w, rs = synth.fp8_weights(N, K, seed=seed, device=DEV)
    x = synth.activations_f16(M, K, seed=seed + 1, device=DEV, outliers=outliers)
    y = q.qgemm_fp8_w8a16(w, rs, x).cpu().numpy()
    rows = np.arange(N) if rows is None else rows
    y_ref, bound = oracle.fp8_w8a16(w.cpu().numpy()[rows], rs.cpu().numpy()[rows], x.cpu().numpy())
    assert_close(f"fp8 M={M} N={N} K={K}", y[:, rows], y_ref, bound)
    return y


@pytest.mark.parametrize("M", range(1, 17))
def test_nvfp4_multi_tile_ragged(q, M):
    q.route_reset()
    _nvfp4(q, M, 16 * 37 + 5, 5120, seed=300 + M)
    assert q.route_counts()["nvfp4_mma_m16n8k16"] == 1


@pytest.mark.parametrize("M", range(1, 17))
def test_fp8_multi_tile_ragged(q, M):
    q.route_reset()
    _fp8(q, M, 16 * 21 + 11, 5120, seed=400 + M)
    assert q.route_counts()["fp8_mma_m16n8k16"] == 1


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 17, 512), (8, 16, 17408), (2, 100, 768),
                                   (9, 100, 768), (12, 33, 512), (16, 16, 17408), (16, 1, 256)])
def test_nvfp4_shapes(q, M, N, K):
    _nvfp4(q, M, N, K, seed=N + K)


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (5, 40, 384), (8, 16, 17408), (2, 31, 1152),
                                   (13, 31, 1152), (16, 40, 384), (16, 16, 17408)])
def test_fp8_shapes(q, M, N, K):
    _fp8(q, M, N, K, seed=N + K)


@pytest.mark.parametrize("M,N,K", [(1, 33, 16), (4, 19, 80), (8, 40, 5136), (11, 19, 80),
                                   (16, 40, 5136)])
def test_nvfp4_generic_k(q, M, N, K):
    q.route_reset()
    _nvfp4(q, M, N, K, seed=K)
    assert q.route_counts()["nvfp4_generic"] == (M + 7) // 8   # one launch per 8 rows


@pytest.mark.parametrize("M,N,K", [(1, 9, 1), (3, 21, 100), (8, 33, 5130), (9, 21, 100), (16, 33, 5130)])
def test_fp8_generic_k(q, M, N, K):
    q.route_reset()
    _fp8(q, M, N, K, seed=K)
    assert q.route_counts()["fp8_generic"] == (M + 7) // 8


@pytest.mark.parametrize("M", [1, 8, 16])
def test_outliers(q, M):
    _nvfp4(q, M, 64, 5120, seed=9, outliers=8)
    _fp8(q, M, 64, 5120, seed=10, outliers=8)


@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("N,K", [(7168, 5120), (5120, 5120), (17408, 5120), (5120, 17408)])
def test_nvfp4_27b_shapes_sampled(q, M, N, K):
    rows = _synth().sample_rows(N, 64, seed=N + K).numpy()
    _nvfp4(q, M, N, K, seed=N * 5 + K + M, rows=rows)


@pytest.mark.parametrize("M", [1, 8, 16])
def test_nvfp4_lm_head_sampled(q, M):
    N, K = 151936, 5120
    rows = _synth().sample_rows(N, 48, seed=M).numpy()
    _nvfp4(q, M, N, K, seed=151936 + M, rows=rows)


@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("N,K", [(7168, 5120), (5120, 5120)])
def test_fp8_27b_attention_shapes_sampled(q, M, N, K):
    rows = _synth().sample_rows(N, 64, seed=N + K + 1).numpy()
    _fp8(q, M, N, K, seed=N * 3 + K + M, rows=rows)


def test_zero_scales(q):
    synth = _synth()
    M, N, K = 3, 48, 2048
    codes, scales, g = synth.nvfp4_weights(N, K, seed=1, device=DEV)
    x = synth.activations_f16(M, K, seed=2, device=DEV)
    scales[7] = 0
    y = q.qgemm_nvfp4_w4a16(codes, scales, g, x)
    assert torch.all(y[:, 7] == 0) and torch.any(y[:, 6] != 0)
    assert torch.all(q.qgemm_nvfp4_w4a16(codes, scales, 0.0, x) == 0)
    w, rs = synth.fp8_weights(N, K, seed=3, device=DEV)
    rs[11] = 0.0
    y = q.qgemm_fp8_w8a16(w, rs, x)
    assert torch.all(y[:, 11] == 0)


def test_unit_codes_closed_form(q):
    """Every code 1.0, every scale 1.0, g = 1: y = sum_k x exactly up to fp32 rounding."""
    M, N, K = 4, 32, 4096
    codes = torch.full((N, K // 2), 0x22, dtype=torch.uint8, device=DEV)
    scales = torch.full((N, K // 16), 0x38, dtype=torch.uint8, device=DEV)
    x = _synth().activations_f16(M, K, seed=5, device=DEV)
    y = q.qgemm_nvfp4_w4a16(codes, scales, 1.0, x).cpu().numpy()
    ref = x.double().sum(dim=1, keepdim=True).expand(M, N).cpu().numpy()
    bound = x.double().abs().sum(dim=1, keepdim=True).expand(M, N).cpu().numpy()
    assert_close("nvfp4 unit codes", y, ref, bound)
    w = torch.full((N, K), 0x38, dtype=torch.uint8, device=DEV)
    y = q.qgemm_fp8_w8a16(w, torch.ones(N, device=DEV), x).cpu().numpy()
    assert_close("fp8 unit codes", y, ref, bound)


def test_k0_and_empty(q):
    x = torch.zeros((2, 0), dtype=torch.float16, device=DEV)
    y = q.qgemm_nvfp4_w4a16(torch.zeros((5, 0), dtype=torch.uint8, device=DEV),
                            torch.zeros((5, 0), dtype=torch.uint8, device=DEV), 1.0, x)
    assert y.shape == (2, 5) and torch.all(y == 0)
    y = q.qgemm_fp8_w8a16(torch.zeros((5, 0), dtype=torch.uint8, device=DEV), torch.ones(5, device=DEV), x)
    assert torch.all(y == 0)


# ------------------------------------------------ grouped launches (one shared x)

@pytest.mark.parametrize("M", [1, 3, 8, 12, 16])
def test_nvfp4_group_matches_oracle(q, M):
    """gate/up-like groups with ragged row counts: every output within the bound."""
    synth = _synth()
    K = 5120
    Ns = [17408, 5120, 37, 1000]
    mats = [synth.nvfp4_weights(n, K, seed=700 + i, device=DEV) for i, n in enumerate(Ns)]
    x = synth.activations_f16(M, K, seed=790, device=DEV, outliers=3)
    q.route_reset()
    outs = q.qgemm_nvfp4_w4a16_group([m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], x)
    assert q.route_counts()["nvfp4_mma_m16n8k16"] == 1
    for i, (c, sc, g) in enumerate(mats):
        rows = np.arange(Ns[i]) if Ns[i] < 2000 else synth.sample_rows(Ns[i], 64, seed=i).numpy()
        y_ref, bound = oracle.nvfp4_w4a16(c.cpu().numpy()[rows], sc.cpu().numpy()[rows], g, x.cpu().numpy())
        assert_close(f"group[{i}]", outs[i].cpu().numpy()[:, rows], y_ref, bound)


@pytest.mark.parametrize("M", [1, 8, 16])
def test_fp8_group_matches_oracle(q, M):
    synth = _synth()
    K = 5120
    Ns = [7168, 5120, 16, 129]
    mats = [synth.fp8_weights(n, K, seed=800 + i, device=DEV) for i, n in enumerate(Ns)]
    x = synth.activations_f16(M, K, seed=890, device=DEV)
    outs = q.qgemm_fp8_w8a16_group([m[0] for m in mats], [m[1] for m in mats], x)
    for i, (w, rs) in enumerate(mats):
        rows = np.arange(Ns[i]) if Ns[i] < 2000 else synth.sample_rows(Ns[i], 64, seed=i).numpy()
        y_ref, bound = oracle.fp8_w8a16(w.cpu().numpy()[rows], rs.cpu().numpy()[rows], x.cpu().numpy())
        assert_close(f"fp8 group[{i}]", outs[i].cpu().numpy()[:, rows], y_ref, bound)


def test_group_of_one_equals_single_call(q):
    """A group of one matrix is the single call (same kernel, same tiles)."""
    synth = _synth()
    c, sc, g = synth.nvfp4_weights(5120, 17408, seed=3, device=DEV)
    x = synth.activations_f16(2, 17408, seed=4, device=DEV)
    assert torch.equal(q.qgemm_nvfp4_w4a16_group([c], [sc], [g], x)[0], q.qgemm_nvfp4_w4a16(c, sc, g, x))


# ------------------------------------------------ 9..16 activation rows

@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("M,K", [(16, 5120), (12, 2048), (9, 17408)])
@pytest.mark.parametrize("staged", [True, False])
def test_two_row_tiles_staged_and_unstaged(q, monkeypatch, fmt, M, K, staged):
    """Activations in shared memory (when they fit) and read through L1: both within the bound."""
    monkeypatch.setenv("QMV_WQ_XSMEM_MAX", str(1 << 20) if staged else "0")
    N = 16 * 45 + 3
    if fmt == "nvfp4":
        _nvfp4(q, M, N, K, seed=950 + M)
    else:
        _fp8(q, M, N, K, seed=960 + M)


def test_rows_beyond_8_do_not_disturb_first_8(q):
    """Rows 1..8 of an M = 16 call agree with the M = 8 call on the same rows (same bound)."""
    synth = _synth()
    codes, scales, g = synth.nvfp4_weights(16 * 30 + 7, 4096, seed=21, device=DEV)
    x = synth.activations_f16(16, 4096, seed=22, device=DEV)
    y16 = q.qgemm_nvfp4_w4a16(codes, scales, g, x).cpu().numpy()
    y8 = q.qgemm_nvfp4_w4a16(codes, scales, g, x[:8].contiguous()).cpu().numpy()
    _, bound = oracle.nvfp4_w4a16(codes.cpu().numpy(), scales.cpu().numpy(), g, x[:8].cpu().numpy())
    assert np.all(np.abs(y16[:8] - y8) <= 2 * (TOL_REL * bound + TOL_ABS))


@pytest.mark.parametrize("fmt,K,passes", [("nvfp4", 4096, 2), ("nvfp4", 4096, 8), ("nvfp4", 17408, 4),
                                          ("fp8", 5120, 5), ("fp8", 1024, 8)])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_k_passes(q, monkeypatch, fmt, K, passes, M):
    """Activations staged one K slice at a time (outputs accumulated over the passes)."""
    monkeypatch.setenv("QMV_WQ_PASSES", str(passes))
    monkeypatch.setenv("QMV_WQ_XSMEM_MAX", str(1 << 20))
    N = 16 * 23 + 9
    if fmt == "nvfp4":
        _nvfp4(q, M, N, K, seed=1000 + M + passes)
    else:
        _fp8(q, M, N, K, seed=1100 + M + passes)


@pytest.mark.parametrize("M", [4, 16])
def test_k_passes_group(q, monkeypatch, M):
    """A gate/up-like group with K cut into passes: each matrix within the bound."""
    monkeypatch.setenv("QMV_WQ_PASSES", "4")
    synth = _synth()
    K = 17408
    Ns = [5120, 40, 1000]
    mats = [synth.nvfp4_weights(n, K, seed=1200 + i, device=DEV) for i, n in enumerate(Ns)]
    x = synth.activations_f16(M, K, seed=1290, device=DEV, outliers=2)
    outs = q.qgemm_nvfp4_w4a16_group([m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], x)
    for i, (c, sc, g) in enumerate(mats):
        rows = np.arange(Ns[i]) if Ns[i] < 2000 else synth.sample_rows(Ns[i], 64, seed=i).numpy()
        y_ref, bound = oracle.nvfp4_w4a16(c.cpu().numpy()[rows], sc.cpu().numpy()[rows], g, x.cpu().numpy())
        assert_close(f"passes group[{i}]", outs[i].cpu().numpy()[:, rows], y_ref, bound)


# ------------------------------------------------ 16-warp CTAs sharing one staged activation copy

@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_sixteen_warps(q, monkeypatch, fmt, M):
    """16 warps per CTA (rounds of 16 interleaved steps, 16-way reduction): within the bound."""
    monkeypatch.setenv("QMV_WQ_WARPS", "16")
    N = 16 * 45 + 3
    if fmt == "nvfp4":
        _nvfp4(q, M, N, 5120, seed=1300 + M)
    else:
        _fp8(q, M, N, 5120, seed=1400 + M)


@pytest.mark.parametrize("passes", [2, 5])
def test_sixteen_warps_passes_group(q, monkeypatch, passes):
    """16 warps, K cut into passes (5 passes: 4 steps per pass, fewer than the warps)."""
    monkeypatch.setenv("QMV_WQ_WARPS", "16")
    monkeypatch.setenv("QMV_WQ_PASSES", str(passes))
    synth = _synth()
    K = 5120
    Ns = [17408, 40, 1000]
    mats = [synth.nvfp4_weights(n, K, seed=1500 + i, device=DEV) for i, n in enumerate(Ns)]
    x = synth.activations_f16(8, K, seed=1590, device=DEV, outliers=2)
    outs = q.qgemm_nvfp4_w4a16_group([m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], x)
    for i, (c, sc, g) in enumerate(mats):
        rows = np.arange(Ns[i]) if Ns[i] < 2000 else synth.sample_rows(Ns[i], 64, seed=i).numpy()
        y_ref, bound = oracle.nvfp4_w4a16(c.cpu().numpy()[rows], sc.cpu().numpy()[rows], g, x.cpu().numpy())
        assert_close(f"16 warps, passes group[{i}]", outs[i].cpu().numpy()[:, rows], y_ref, bound)


# ------------------------------------------------ 17..96 rows: balanced chunks of <= 16 rows

@pytest.fixture
def chunked(monkeypatch):
    """The chunked mma.sync path above 16 rows (the tcgen05 kernel switched off)."""
    monkeypatch.setenv("QMV_WQ_UMMA_MIN_M", "0")


@pytest.mark.parametrize("M", [17, 24, 33, 64, 96])
def test_chunked_rows(q, M, chunked):
    """ceil(M / 16) launches of <= 16 rows each; every output within the bound."""
    N = 16 * 21 + 11
    q.route_reset()
    _nvfp4(q, M, N, 5120, seed=1600 + M)
    _fp8(q, M, N, 5120, seed=1700 + M)
    c = q.route_counts()
    assert c["nvfp4_mma_m16n8k16"] == (M + 15) // 16 and c["fp8_mma_m16n8k16"] == (M + 15) // 16


@pytest.mark.parametrize("M", [40, 96])
@pytest.mark.parametrize("N,K", [(7168, 5120), (5120, 5120)])
def test_fp8_chunked_27b_attention_sampled(q, M, N, K, chunked):
    rows = _synth().sample_rows(N, 24, seed=N + K + M).numpy()
    _fp8(q, M, N, K, seed=N * 11 + K + M, rows=rows)


@pytest.mark.parametrize("M", [17, 96])
def test_chunked_group_and_generic(q, M, chunked):
    """A gate/up-like group chunked by rows, and the generic kernel (K % 256 != 0) at M > 16."""
    synth = _synth()
    K = 5120
    Ns = [1000, 40]
    mats = [synth.nvfp4_weights(n, K, seed=1800 + i, device=DEV) for i, n in enumerate(Ns)]
    x = synth.activations_f16(M, K, seed=1890, device=DEV, outliers=2)
    outs = q.qgemm_nvfp4_w4a16_group([m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], x)
    for i, (c, sc, g) in enumerate(mats):
        y_ref, bound = oracle.nvfp4_w4a16(c.cpu().numpy(), sc.cpu().numpy(), g, x.cpu().numpy())
        assert_close(f"chunked group[{i}]", outs[i].cpu().numpy(), y_ref, bound)
    q.route_reset()
    _nvfp4(q, M, 33, 1040, seed=1900 + M)
    _fp8(q, M, 21, 1000, seed=1950 + M)
    assert q.route_counts()["nvfp4_generic"] == (M + 7) // 8 and q.route_counts()["fp8_generic"] == (M + 7) // 8


@pytest.mark.parametrize("M", [8, 9, 16, 17, 32, 96])
@pytest.mark.parametrize("N", [128 * 2 + 45, 128 * 60 + 7])
def test_default_dispatch(q, monkeypatch, M, N):
    """Default routes: one mma.sync pass up to 8 rows; from 9 rows the tcgen05 kernel
    (one launch, one weight pass, K split over a cluster) when the launch has at most a
    third of the SMs' worth of 128-row tiles (3 tiles here); otherwise (61 tiles) mma.sync
    up to 16 rows and the tcgen05 kernel from 17, for NVFP4 and FP8 alike."""
    monkeypatch.delenv("QMV_WQ_UMMA_FEW_TILES_MIN_M", raising=False)
    few = (N + 127) // 128 * 3 <= 152
    umma = M >= 17 or (few and M >= 9)
    rows = np.arange(N) if N < 1000 else _synth().sample_rows(N, 48, seed=N + M).numpy()
    q.route_reset()
    _nvfp4(q, M, N, 5120, seed=3100 + M, rows=rows)
    _fp8(q, M, N, 5120, seed=3200 + M, rows=rows)
    c = {k: v for k, v in q.route_counts().items() if v}
    want = {"nvfp4_tcgen05": 1, "fp8_tcgen05": 1} if umma else {"nvfp4_mma_m16n8k16": 1, "fp8_mma_m16n8k16": 1}
    assert c == want, c
    for fp4 in (True, False):
        assert q.qmv_debug_plan_wq(M, 5120, [N], fp4=fp4)["route"] == ("nvfp4" if fp4 else "fp8") + (
            "_tcgen05" if umma else "_mma_m16n8k16")


# ------------------------------------------------ largest K and M

@pytest.mark.parametrize("M", [1, 8, 16])
def test_nvfp4_large_k(q, M):
    """K = 65536 (a 2 MB fp16 activation matrix at M = 16): staged in passes or read
    through L1, within the bound."""
    _nvfp4(q, M, 16 * 7 + 3, 65536, seed=2300 + M, outliers=2)


def test_fp8_largest_m_large_k(q):
    """M = 96 (six 16-row chunks) with K = 16384."""
    _fp8(q, 96, 16 * 5 + 1, 16384, seed=2400)

"""GPU parity of the tcgen05 NVFP4 / FP8 kernel (wq_umma.cu) against the CPU oracle.

The kernel computes the products of "v100-skinny README", section "How QPN works"
(QPN2: NVFP4 W4A16; QPN8: FP8 W8A16) with tcgen05.mma: 128 weight rows per tile in
tensor memory, all M <= 96 activation rows (zero-padded to a multiple of 16) in one
pass over the weights. QMV_WQ_UMMA_MIN_M=1 routes every aligned call to it here.
Every fp32 output within |y - y_ref| <= 1e-3 * sum|w*x| + 1e-6 on: tiles with a
ragged tail (N not a multiple of 128) at M = 1..96 including every padding boundary,
K from one step to 17408, fp16 outliers up to 6e4, zero scales, the closed form of
unit codes, groups with ragged row counts, and sampled rows of the 27B-class shapes
and the 151936-row lm_head; split K (clusters of 2..4 CTAs per tile, partial sums
added in the rank-0 CTA) forced on and off on the same inputs. The route census must
show the tcgen05 route only.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def q():
    from gemm_qmv_quantize_gb300 import build
    build.build()
    import gemm_qmv_quantize_gb300 as q
    return q


@pytest.fixture(autouse=True)
def umma_on(monkeypatch):
    monkeypatch.setenv("QMV_WQ_UMMA_MIN_M", "1")


def _synth():
    from gemm_qmv_quantize_gb300 import synth
    return synth


def _nvfp4(q, M, N, K, seed, outliers=0, rows=None):
    synth = _synth()
    codes, scales, g = synth.nvfp4_weights(N, K, seed=seed, device=DEV)
    x = synth.activations_f16(M, K, seed=seed + 1, device=DEV, outliers=outliers)
    q.route_reset()
    y = q.qgemm_nvfp4_w4a16(codes, scales, g, x).cpu().numpy()
    assert {k: v for k, v in q.route_counts().items() if v} == {"nvfp4_tcgen05": 1}
    rows = np.arange(N) if rows is None else rows
    y_ref, bound = oracle.nvfp4_w4a16(codes.cpu().numpy()[rows], scales.cpu().numpy()[rows], g, x.cpu().numpy())
    assert_close(f"nvfp4 tcgen05 M={M} N={N} K={K}", y[:, rows], y_ref, bound)
    assert q.error_flags() == 0


def _fp8(q, M, N, K, seed, outliers=0, rows=None):
    synth = _synth()
    w, rs = synth.fp8_weights(N, K, seed=seed, device=DEV)
    x = synth.activations_f16(M, K, seed=seed + 1, device=DEV, outliers=outliers)
    q.route_reset()
    y = q.qgemm_fp8_w8a16(w, rs, x).cpu().numpy()
    assert {k: v for k, v in q.route_counts().items() if v} == {"fp8_tcgen05": 1}
    rows = np.arange(N) if rows is None else rows
    y_ref, bound = oracle.fp8_w8a16(w.cpu().numpy()[rows], rs.cpu().numpy()[rows], x.cpu().numpy())
    assert_close(f"fp8 tcgen05 M={M} N={N} K={K}", y[:, rows], y_ref, bound)
    assert q.error_flags() == 0


def test_first_small_case(q):
    _nvfp4(q, 1, 128, 256, seed=1)
    _fp8(q, 1, 128, 128, seed=2)


@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64, 80, 95, 96])
def test_nvfp4_ragged_tiles(q, M):
    _nvfp4(q, M, 128 * 3 + 37, 5120, seed=1000 + M)


@pytest.mark.parametrize("M", [1, 2, 8, 9, 16, 17, 32, 33, 64, 96])
def test_fp8_ragged_tiles(q, M):
    _fp8(q, M, 128 * 2 + 91, 5120, seed=2000 + M)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 129, 512), (16, 300, 17408), (40, 5, 768), (96, 257, 1024)])
def test_nvfp4_shapes(q, M, N, K):
    _nvfp4(q, M, N, K, seed=N + K + M)


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (5, 130, 384), (16, 77, 17408), (33, 200, 1152), (96, 128, 640)])
def test_fp8_shapes(q, M, N, K):
    _fp8(q, M, N, K, seed=N + K + M)


@pytest.mark.parametrize("M", [1, 16, 96])
def test_outliers(q, M):
    _nvfp4(q, M, 256, 5120, seed=9, outliers=8)
    _fp8(q, M, 256, 5120, seed=10, outliers=8)


@pytest.mark.parametrize("M", [1, 8, 16, 32, 96])
@pytest.mark.parametrize("N,K", [(7168, 5120), (5120, 5120), (17408, 5120), (5120, 17408)])
def test_nvfp4_27b_shapes_sampled(q, M, N, K):
    rows = _synth().sample_rows(N, 64, seed=N + K).numpy()
    _nvfp4(q, M, N, K, seed=N * 7 + K + M, rows=rows)


@pytest.mark.parametrize("M", [1, 16, 96])
@pytest.mark.parametrize("N,K", [(7168, 5120), (5120, 5120)])
def test_fp8_27b_attention_shapes_sampled(q, M, N, K):
    rows = _synth().sample_rows(N, 64, seed=N + K + 3).numpy()
    _fp8(q, M, N, K, seed=N * 11 + K + M, rows=rows)


@pytest.mark.parametrize("M", [1, 16])
def test_nvfp4_lm_head_sampled(q, M):
    N, K = 151936, 5120
    rows = _synth().sample_rows(N, 48, seed=M + 5).numpy()
    _nvfp4(q, M, N, K, seed=151936 + 3 * M, rows=rows)


def test_zero_scales_and_unit_codes(q):
    synth = _synth()
    M, N, K = 3, 160, 2048
    codes, scales, g = synth.nvfp4_weights(N, K, seed=1, device=DEV)
    x = synth.activations_f16(M, K, seed=2, device=DEV)
    scales[7] = 0
    y = q.qgemm_nvfp4_w4a16(codes, scales, g, x)
    assert torch.all(y[:, 7] == 0) and torch.any(y[:, 6] != 0)
    w, rs = synth.fp8_weights(N, K, seed=3, device=DEV)
    rs[130] = 0.0
    assert torch.all(q.qgemm_fp8_w8a16(w, rs, x)[:, 130] == 0)
    # every code 1.0, every scale 1.0, g = 1: y = sum_k x up to fp32 rounding
    M, N, K = 20, 130, 4096
    codes = torch.full((N, K // 2), 0x22, dtype=torch.uint8, device=DEV)
    scales = torch.full((N, K // 16), 0x38, dtype=torch.uint8, device=DEV)
    x = synth.activations_f16(M, K, seed=5, device=DEV)
    y = q.qgemm_nvfp4_w4a16(codes, scales, 1.0, x).cpu().numpy()
    ref = x.double().sum(dim=1, keepdim=True).expand(M, N).cpu().numpy()
    bound = x.double().abs().sum(dim=1, keepdim=True).expand(M, N).cpu().numpy()
    assert_close("nvfp4 tcgen05 unit codes", y, ref, bound)
    wq = torch.full((N, K), 0x38, dtype=torch.uint8, device=DEV)
    assert_close("fp8 tcgen05 unit codes", q.qgemm_fp8_w8a16(wq, torch.ones(N, device=DEV), x).cpu().numpy(), ref,
                 bound)


@pytest.mark.parametrize("M", [1, 9, 40])
def test_groups(q, M):
    """A group of 136 + 40 + 1 + 8 = 185 tiles on 152 CTAs: 33 CTAs take a second tile.
    At M = 40 the plan has T = 3 issuing threads and 80 quarters per tile, not a
    multiple of 3, so a tile's first A buffers change issuing thread at the boundary
    (ordered by the wait for the previous tile's read-back)."""
    synth = _synth()
    K = 5120
    Ns = [17408, 5120, 37, 1000]
    mats = [synth.nvfp4_weights(n, K, seed=900 + i, device=DEV) for i, n in enumerate(Ns)]
    x = synth.activations_f16(M, K, seed=990, device=DEV, outliers=3)
    q.route_reset()
    outs = q.qgemm_nvfp4_w4a16_group([m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], x)
    assert {k: v for k, v in q.route_counts().items() if v} == {"nvfp4_tcgen05": 1}
    for i, (c, sc, g) in enumerate(mats):
        rows = np.arange(Ns[i]) if Ns[i] < 2000 else synth.sample_rows(Ns[i], 64, seed=i).numpy()
        y_ref, bound = oracle.nvfp4_w4a16(c.cpu().numpy()[rows], sc.cpu().numpy()[rows], g, x.cpu().numpy())
        assert_close(f"tcgen05 group[{i}]", outs[i].cpu().numpy()[:, rows], y_ref, bound)
    wm = [synth.fp8_weights(n, K, seed=950 + i, device=DEV) for i, n in enumerate([7168, 5120])]
    outs = q.qgemm_fp8_w8a16_group([m[0] for m in wm], [m[1] for m in wm], x)
    for i, (w, rs) in enumerate(wm):
        rows = synth.sample_rows(w.shape[0], 64, seed=i + 7).numpy()
        y_ref, bound = oracle.fp8_w8a16(w.cpu().numpy()[rows], rs.cpu().numpy()[rows], x.cpu().numpy())
        assert_close(f"tcgen05 fp8 group[{i}]", outs[i].cpu().numpy()[:, rows], y_ref, bound)


@pytest.mark.parametrize("M", [9, 33, 96])
def test_groups_split_k(q, M):
    """Grouped launches of few tiles: the cluster's CTAs share a tile of any matrix of
    the group (NVFP4: 8 + 1 + 5 + 16 tiles, 4 CTAs per tile; FP8: 40 + 3 tiles, 3 per
    tile), every output within the bound."""
    synth = _synth()
    K = 5120
    Ns = [1000, 37, 513, 2048]
    assert q.qmv_debug_plan_wq(M, K, Ns, fp4=True)["k_splits"] == 4
    mats = [synth.nvfp4_weights(n, K, seed=1200 + i, device=DEV) for i, n in enumerate(Ns)]
    x = synth.activations_f16(M, K, seed=1290 + M, device=DEV, outliers=2)
    q.route_reset()
    outs = q.qgemm_nvfp4_w4a16_group([m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], x)
    assert {k: v for k, v in q.route_counts().items() if v} == {"nvfp4_tcgen05": 1}
    for i, (c, sc, g) in enumerate(mats):
        y_ref, bound = oracle.nvfp4_w4a16(c.cpu().numpy(), sc.cpu().numpy(), g, x.cpu().numpy())
        assert_close(f"split group[{i}] M={M}", outs[i].cpu().numpy(), y_ref, bound)
    Nf = [5120, 300]
    assert q.qmv_debug_plan_wq(M, K, Nf, fp4=False)["k_splits"] == 3
    wm = [synth.fp8_weights(n, K, seed=1250 + i, device=DEV) for i, n in enumerate(Nf)]
    outs = q.qgemm_fp8_w8a16_group([m[0] for m in wm], [m[1] for m in wm], x)
    for i, (w, rs) in enumerate(wm):
        rows = np.arange(w.shape[0]) if w.shape[0] < 1000 else synth.sample_rows(w.shape[0], 96, seed=i + M).numpy()
        y_ref, bound = oracle.fp8_w8a16(w.cpu().numpy()[rows], rs.cpu().numpy()[rows], x.cpu().numpy())
        assert_close(f"split fp8 group[{i}] M={M}", outs[i].cpu().numpy()[:, rows], y_ref, bound)
    assert q.error_flags() == 0


def test_chain_with_launch_overlap(q):
    """Back-to-back calls with programmatic dependent launch (as the stacks run them):
    each call's outputs match the oracle (the next call's weight copies start while
    the previous one drains; tensor memory is allocated per CTA)."""
    synth = _synth()
    before = q.get_launch_overlap()
    q.set_launch_overlap(True)
    try:
        K = 5120
        mats = [synth.nvfp4_weights(5120, K, seed=1100 + i, device=DEV) for i in range(4)]
        x = synth.activations_f16(16, K, seed=1190, device=DEV)
        ys = [q.qgemm_nvfp4_w4a16(c, sc, g, x) for c, sc, g in mats]
        torch.cuda.synchronize()
        for i, (c, sc, g) in enumerate(mats):
            rows = synth.sample_rows(5120, 64, seed=i + 11).numpy()
            y_ref, bound = oracle.nvfp4_w4a16(c.cpu().numpy()[rows], sc.cpu().numpy()[rows], g, x.cpu().numpy())
            assert_close(f"chain[{i}]", ys[i].cpu().numpy()[:, rows], y_ref, bound)
    finally:
        q.set_launch_overlap(before)


@pytest.mark.parametrize("fp4", [True, False])
@pytest.mark.parametrize("splits", [1, 2, 3, 4])
def test_split_k_forced(q, monkeypatch, fp4, splits):
    """The same call with the K range split over 1..4 CTAs of a cluster: every split
    count within the bound against the oracle, on a ragged tile count and a K whose
    steps do not divide evenly between the CTAs (K = 5120: 20 NVFP4 / 40 FP8 steps)."""
    monkeypatch.setenv("QMV_UMMA_SPLITS", str(splits))
    M, N, K = 33, 1000, 5120
    assert q.qmv_debug_plan_wq(M, K, [N], fp4=fp4)["k_splits"] == splits
    (_nvfp4 if fp4 else _fp8)(q, M, N, K, seed=700 + splits + (0 if fp4 else 50))


def test_split_k_default_on_few_tiles(q):
    """With few tiles the default plan splits K (40 tiles of the 5120-row matrices: 3
    CTAs each) and the result stays within the bound on sampled rows of every tile."""
    M, N, K = 32, 5120, 17408
    assert q.qmv_debug_plan_wq(M, K, [N], fp4=True)["k_splits"] == 3
    rows = np.unique(np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128)]))
    _nvfp4(q, M, N, K, seed=4242, rows=rows)

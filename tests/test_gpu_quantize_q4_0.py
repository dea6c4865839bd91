"""GPU parity: Q8_1 quantizer and Q4_0 x Q8_1 MMVQ through the C ABI vs the CPU oracle.

- Q8_1 bytes (d8, s8, q) identical to the oracle's.
- Integer block sums S - 8T identical (qmv_debug_q4_0_block_dots runs the
  product kernel's device code with the product kernel choice).
- fp32 outputs within |y - y_ref| <= 1e-3 * sum|w*x| + 1e-6.
Shapes span several tiles with a ragged tail, M = 1..8, the streaming and the
generic kernels, and the full-size matrices of the Llama-2-7B and Llama-3-8B
shaped workloads (sampled rows).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import GOLDEN
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def q():
    from gemm_qmv_quantize_gb300 import build
    build.build()
    import gemm_qmv_quantize_gb300 as q
    return q


def _synth():
    from gemm_qmv_quantize_gb300 import synth
    return synth


# ---------------------------------------------------------------- quantizer

@pytest.mark.parametrize("M,K", [(1, 32), (1, 4096), (3, 11008), (8, 14336), (2, 4128)])
def test_quantize_bytes_exact(q, M, K):
    x = _synth().activations_f32(M, K, seed=M * 7 + K, device=DEV)
    x[0, :32] *= 1e-30        # subnormal-range scale
    if K >= 64:
        x[0, 32:64] = 0.0     # all-zero block
    xq = q.qmv_quantize_q8_1(x)
    ref = oracle.quantize_q8_1(x.cpu().numpy())
    assert np.array_equal(xq.cpu().numpy(), ref)


def test_quantize_golden_blocks(q):
    with open(os.path.join(GOLDEN, "q8_1_blocks.json")) as f:
        cases = json.load(f)["cases"]
    by = {c["name"]: c for c in cases}
    rows = []
    for c in cases:
        x = np.array(c["x"] if "x" in c else by[c["x_from"]]["x"], dtype=np.float32)
        if "x_scale" in c:
            x = x * np.float32(c["x_scale"])
        rows.append(x)
    x = torch.from_numpy(np.concatenate(rows)[None, :]).to(DEV)
    xq = q.qmv_quantize_q8_1(x).cpu().numpy().reshape(-1, 36)
    for i, c in enumerate(cases):
        d8 = int(xq[i, 0]) | int(xq[i, 1]) << 8
        s8 = int(xq[i, 2]) | int(xq[i, 3]) << 8
        assert list(xq[i, 4:].view(np.int8)) == c["q"], c["name"]
        assert d8 == int(c["d8"], 16) and s8 == int(c["s8"], 16), c["name"]


def test_quantize_ties_and_extremes(q):
    """Elements landing exactly on k + 1/2 after the division, and large magnitudes."""
    K = 32 * 64
    rng = np.random.default_rng(3)
    x = np.empty((2, K), np.float32)
    for b in range(64):
        blk = (rng.integers(-254, 255, 32) / 2.0).astype(np.float32)   # multiples of 1/2
        blk[0] = 127.0                                                  # d = 1 -> ties at .5
        x[0, 32 * b:32 * (b + 1)] = blk * np.float32(2.0 ** (b % 9 - 4))
    x[1] = (rng.standard_normal(K) * 1e5).astype(np.float32)
    xt = torch.from_numpy(x).to(DEV)
    assert np.array_equal(q.qmv_quantize_q8_1(xt).cpu().numpy(), oracle.quantize_q8_1(x))


def test_quantize_near_ties(q):
    """Values within a few ulps of k + 1/2 after the division, at scales whose
    reciprocal is inexact: the kernels must take every rounding decision as the
    correctly rounded fp32 quotient does."""
    rng = np.random.default_rng(17)
    nblk = 2048
    x = np.zeros((1, 32 * nblk), np.float32)
    for bi in range(nblk):
        amax = np.float32(rng.uniform(0.01, 100.0))
        d = np.float32(amax / np.float32(127.0))
        blk = np.empty(32, np.float32)
        blk[0] = amax if bi % 2 else -amax
        k = rng.integers(-126, 126, 31).astype(np.float32)
        t = (k + np.float32(0.5)) * d                      # near a tie after x / d
        steps = rng.integers(-3, 4, 31)
        blk[1:] = np.array([np.nextafter(tv, np.float32(np.inf) if st > 0 else np.float32(-np.inf))
                            if st else tv for tv, st in zip(t, steps)], np.float32)
        for _ in range(2):   # up to a few more ulps
            blk[1:] = np.where(steps > 1, np.nextafter(blk[1:], np.float32(np.inf)), blk[1:])
            blk[1:] = np.where(steps < -1, np.nextafter(blk[1:], np.float32(-np.inf)), blk[1:])
        np.clip(blk, -amax, amax, out=blk)
        x[0, 32 * bi:32 * (bi + 1)] = blk
    xt = torch.from_numpy(x).to(DEV)
    ref = oracle.quantize_q8_1(x)
    assert np.array_equal(q.qmv_quantize_q8_1(xt).cpu().numpy(), ref)
    # the fused prologue takes the same decisions: compare against the two-call path
    from gemm_qmv_quantize_gb300 import synth
    K = x.shape[1]
    w = synth.q4_0_weights(64, K, seed=3, device=DEV)
    assert torch.equal(q.qmv_q4_0_q8_1_fused(w, xt), q.qmv_q4_0_q8_1(w, torch.from_numpy(ref).to(DEV), K))


# ---------------------------------------------------------------- Q4_0 MMVQ

def _q4_case(q, M, N, K, seed, offset=0):
    synth = _synth()
    w = synth.q4_0_weights(N, K, seed=seed, device=DEV)
    if offset:
        # same bytes at a 2-byte (not 16-byte) aligned address: the generic kernel
        buf = torch.empty(w.numel() + 16, dtype=torch.uint8, device=DEV)
        buf[offset:offset + w.numel()] = w.view(-1)
        w = buf[offset:offset + w.numel()].view(N, -1)
    x = synth.activations_f32(M, K, seed=seed + 1, device=DEV)
    xq = q.qmv_quantize_q8_1(x)
    return w, xq


def _check_q4(q, M, N, K, seed, offset=0, full=True, rows=None):
    w, xq = _q4_case(q, M, N, K, seed, offset)
    if offset:
        from gemm_qmv_quantize_gb300 import _binding
        y = torch.empty((M, N), dtype=torch.float32, device=DEV)
        dots = torch.empty((M, N, K // 32), dtype=torch.int32, device=DEV)
        L = _binding.lib()
        s = torch.cuda.current_stream().cuda_stream
        assert L.qmv_q4_0_q8_1(w.data_ptr(), xq.data_ptr(), y.data_ptr(), M, N, K, s) == 0
        assert L.qmv_debug_q4_0_block_dots(w.data_ptr(), xq.data_ptr(), dots.data_ptr(), M, N, K, s) == 0
    else:
        y = q.qmv_q4_0_q8_1(w, xq, K)
        dots = q.qmv_debug_q4_0_block_dots(w, xq, K)
    torch.cuda.synchronize()
    wn = w.cpu().numpy()
    xqn = xq.cpu().numpy()
    if rows is None:
        rows = np.arange(N)
    S, T = oracle.q4_0_block_dots(np.ascontiguousarray(wn[rows]), xqn, K)
    assert np.array_equal(dots.cpu().numpy()[:, rows, :], S - 8 * T[:, None, :]), "integer block sums"
    y_ref, bound = oracle.q4_0_q8_1(np.ascontiguousarray(wn[rows]), xqn, K)
    assert_close(f"q4_0 M={M} N={N} K={K}", y.cpu().numpy()[:, rows], y_ref, bound)


@pytest.mark.parametrize("M", range(1, 9))
def test_q4_0_multi_tile_ragged(q, M):
    _check_q4(q, M, 1000 + M, 4096, seed=100 + M)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 37, 256), (1, 5, 512), (3, 300, 11008), (8, 130, 14336),
                                   (1, 2049, 768)])
def test_q4_0_shapes(q, M, N, K):
    _check_q4(q, M, N, K, seed=N + K)


@pytest.mark.parametrize("M,N,K", [(1, 33, 96), (4, 70, 4128), (8, 9, 32)])
def test_q4_0_generic_k(q, M, N, K):
    q.route_reset()
    _check_q4(q, M, N, K, seed=K)
    assert q.route_counts()["q4_0_generic"] > 0


def test_q4_0_unaligned_rows_use_generic_kernel(q):
    q.route_reset()
    _check_q4(q, 2, 200, 4096, seed=5, offset=2)
    rc = q.route_counts()
    assert rc["q4_0_generic"] == 2 and rc["q4_0_stream_dp4a"] == 0


def test_q4_0_full_4096_square(q):
    """The small single-matrix workload: M = 1, N = K = 4096, every output checked."""
    q.route_reset()
    _check_q4(q, 1, 4096, 4096, seed=2024)
    assert q.route_counts()["q4_0_stream_dp4a"] == 2


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("N,K", [(11008, 4096), (4096, 11008), (32000, 4096)])
def test_q4_0_llama2_7b_shapes_sampled(q, M, N, K):
    from gemm_qmv_quantize_gb300 import synth
    rows = synth.sample_rows(N, 96, seed=N).numpy()
    _check_q4(q, M, N, K, seed=N * 3 + K, rows=rows)


@pytest.mark.parametrize("M", range(1, 9))
@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_q4_0_llama3_8b_mlp_sampled(q, M, N, K):
    from gemm_qmv_quantize_gb300 import synth
    rows = synth.sample_rows(N, 48, seed=N + M).numpy()
    _check_q4(q, M, N, K, seed=N + 7 * K + M, rows=rows)


def test_q4_0_special_weights(q):
    """Zero scales give zero rows; all-8 nibbles give exact zeros."""
    M, N, K = 2, 64, 4096
    w, xq = _q4_case(q, M, N, K, seed=77)
    blk = w.view(N, K // 32, 18)
    blk[3, :, 0:2] = 0
    blk[5, :, 2:] = 0x88
    y = q.qmv_q4_0_q8_1(w, xq, K).cpu().numpy()
    assert np.all(y[:, 3] == 0.0) and np.all(y[:, 5] == 0.0)


def test_q4_0_empty_and_k0(q):
    x = torch.zeros((1, 0), dtype=torch.float32, device=DEV)
    w = torch.zeros((4, 0), dtype=torch.uint8, device=DEV)
    xq = torch.zeros((1, 0), dtype=torch.uint8, device=DEV)
    assert q.qmv_quantize_q8_1(x).numel() == 0
    y = torch.full((1, 4), 7.0, device=DEV)
    q.qmv_q4_0_q8_1(w, xq, 0, out=y)
    assert torch.all(y == 0)
    w0 = torch.zeros((0, 4096 // 32 * 18), dtype=torch.uint8, device=DEV)
    xq0 = torch.zeros((1, 4096 // 32 * 36), dtype=torch.uint8, device=DEV)
    assert q.qmv_q4_0_q8_1(w0, xq0, 4096).shape == (1, 0)


def test_launch_overlap_chain_matches_plain(q):
    """A dependent chain of calls (each activation produced by the previous call's
    output, as in decode) gives bit-identical results with launch overlap on."""
    from gemm_qmv_quantize_gb300 import synth
    shapes = [(4096, 4096), (11008, 4096), (4096, 11008), (4096, 4096)]
    ws = [synth.q4_0_weights(n, k, seed=50 + i, device=DEV) for i, (n, k) in enumerate(shapes)]
    x0 = synth.activations_f32(1, 4096, seed=49, device=DEV)

    def chain():
        x = x0
        outs = []
        for (n, k), w in zip(shapes, ws):
            xin = x[:, :k] if x.shape[1] >= k else x.repeat(1, (k + x.shape[1] - 1) // x.shape[1])[:, :k]
            xin = xin.contiguous()
            y = q.qmv_q4_0_q8_1(w, q.qmv_quantize_q8_1(xin), k)
            outs.append(y)
            x = y
        return [o.clone() for o in outs]

    prev = q.get_launch_overlap()
    try:
        q.set_launch_overlap(False)
        plain = chain()
        q.set_launch_overlap(True)
        over = chain()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            graphed = chain()
        g.replay()
        torch.cuda.synchronize()
    finally:
        q.set_launch_overlap(prev)
    for a, b, c in zip(plain, over, graphed):
        assert torch.equal(a, b) and torch.equal(a, c)
    # and the chain itself is right: check the first call against the oracle
    xq_ref = oracle.quantize_q8_1(x0.cpu().numpy())
    y_ref, bound = oracle.q4_0_q8_1(ws[0].cpu().numpy(), xq_ref, 4096)
    assert_close("chain[0]", plain[0].cpu().numpy(), y_ref, bound)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (3, 1000, 11008), (8, 300, 14336), (2, 37, 256),
                                   (1, 32000, 4096), (5, 777, 4096)])
def test_q4_0_fused_matches_two_calls(q, M, N, K):
    """Quantize-in-prologue gives bit-identical outputs to quantize + MMVQ, and meets the oracle."""
    from gemm_qmv_quantize_gb300 import synth
    w = synth.q4_0_weights(N, K, seed=N + K + M, device=DEV)
    x = synth.activations_f32(M, K, seed=N + K + M + 1, device=DEV)
    x[0, :32] *= 1e-30
    q.route_reset()
    y2 = q.qmv_q4_0_q8_1(w, q.qmv_quantize_q8_1(x), K)
    y1 = q.qmv_q4_0_q8_1_fused(w, x)
    assert torch.equal(y1, y2)
    rc = q.route_counts()
    assert rc["q4_0_stream_fused_quantize"] + rc["q4_0_mma_fused_quantize"] == 1
    rows = synth.sample_rows(N, 64, seed=M).numpy()
    xq_ref = oracle.quantize_q8_1(x.cpu().numpy())
    y_ref, bound = oracle.q4_0_q8_1(np.ascontiguousarray(w.cpu().numpy()[rows]), xq_ref, K)
    assert_close("fused", y1.cpu().numpy()[:, rows], y_ref, bound)


def test_q4_0_fused_rejects_unsupported_shapes(q):
    from gemm_qmv_quantize_gb300 import QmvError, synth
    w = synth.q4_0_weights(8, 96, seed=1, device=DEV)
    x = synth.activations_f32(1, 96, seed=2, device=DEV)
    with pytest.raises(QmvError, match="SHAPE"):
        q.qmv_q4_0_q8_1_fused(w, x)
    w = synth.q4_0_weights(8, 512, seed=1, device=DEV)
    buf = torch.empty(w.numel() + 16, dtype=torch.uint8, device=DEV)
    wm = buf[2:2 + w.numel()].view(8, -1)
    with pytest.raises(QmvError, match="ALIGN"):
        q.qmv_q4_0_q8_1_fused(wm, synth.activations_f32(1, 512, seed=2, device=DEV))


@pytest.mark.parametrize("M,pattern", [(1, (0, 0, 1, 1)), (3, (0, 0, 1, 1)), (8, (0, 0, 1, 1)),
                                       (1, (0, 1, 2, 3)), (1, (0, 1, 0, 2)), (4, (2, 0, 2, 1))])
def test_q4_0_fused_group_matches_single_calls(q, M, pattern):
    """A grouped launch of independent matrices (q/k/v-like; matrices given the same
    input tensor share its staging) is bit-identical to one fused call per matrix."""
    from gemm_qmv_quantize_gb300 import synth
    K = 4096
    Ns = [4096, 1024, 1024, 11008]
    ws = [synth.q4_0_weights(n, K, seed=900 + i, device=DEV) for i, n in enumerate(Ns)]
    inputs = [synth.activations_f32(M, K, seed=990 + j, device=DEV) for j in range(max(pattern) + 1)]
    xs = [inputs[j] for j in pattern]
    xb = xs[3]
    q.route_reset()
    outs = q.qmv_q4_0_q8_1_fused_group(ws, xs)
    singles = [q.qmv_q4_0_q8_1_fused(w, x) for w, x in zip(ws, xs)]
    for a, b in zip(outs, singles):
        assert torch.equal(a, b)
    rc = q.route_counts()
    assert rc["q4_0_stream_fused_quantize"] + rc["q4_0_mma_fused_quantize"] == 5
    rows = synth.sample_rows(Ns[3], 32, seed=M).numpy()
    y_ref, bound = oracle.q4_0_q8_1(np.ascontiguousarray(ws[3].cpu().numpy()[rows]),
                                    oracle.quantize_q8_1(xb.cpu().numpy()), K)
    assert_close("group[3]", outs[3].cpu().numpy()[:, rows], y_ref, bound)


def test_q4_0_fused_group_validation(q):
    from gemm_qmv_quantize_gb300 import _binding
    L = _binding.lib()
    import ctypes
    P = ctypes.c_void_p * 9
    n = (ctypes.c_int64 * 9)(*([64] * 9))
    z = P(*([0x10000] * 9))
    assert L.qmv_q4_0_q8_1_fused_group(9, z, z, z, n, 1, 4096, None) == -2     # count > 8
    assert L.qmv_q4_0_q8_1_fused_group(0, z, z, z, n, 1, 4096, None) == -2
    assert L.qmv_q4_0_q8_1_fused_group(2, z, z, z, n, 1, 4000, None) == -2     # K % 256
    bad = P(0x10000, 0x10008)
    assert L.qmv_q4_0_q8_1_fused_group(2, bad, z, z, n, 1, 4096, None) == -3   # w not 16-aligned


# ------------------------------------------------ the two Q4_0 kernels at M >= 2

@pytest.fixture(params=["mma", "dp4a"])
def q4_kernel(request, monkeypatch):
    """Route M >= 2 to the tensor-core kernel or to the dp4a streaming kernel (the
    planner's minimum M for the tensor cores set to 2, or raised past 8)."""
    monkeypatch.setenv("QMV_Q4_MMA_MIN_M", "9" if request.param == "dp4a" else "2")
    return request.param


@pytest.mark.parametrize("M,N,K", [(2, 1000, 4096), (3, 37, 256), (4, 300, 11008), (5, 129, 768),
                                   (6, 16, 14336), (7, 513, 4096), (8, 1000, 4096), (8, 77, 512)])
def test_q4_0_both_kernels_match_oracle(q, q4_kernel, M, N, K):
    """Integer block sums bit-exact and outputs within the bound on either kernel,
    over ragged tiles, every tile-round shape (K / 256 steps of 1, 2, 3, 16, 43, 56)."""
    q.route_reset()
    _check_q4(q, M, N, K, seed=7 * N + K + M)
    rc = q.route_counts()
    want = "q4_0_mma_m16n8k32" if q4_kernel == "mma" else "q4_0_stream_dp4a"
    assert rc[want] == 2, rc


@pytest.mark.parametrize("M", [2, 5, 8])
def test_q4_0_fused_group_both_kernels(q, q4_kernel, M):
    """Grouped, fused launches (shared and distinct inputs) agree with single calls on either kernel."""
    from gemm_qmv_quantize_gb300 import synth
    K = 4096
    Ns = [1024, 4096, 1000, 16]
    ws = [synth.q4_0_weights(n, K, seed=1900 + i, device=DEV) for i, n in enumerate(Ns)]
    inputs = [synth.activations_f32(M, K, seed=1990 + j, device=DEV) for j in range(2)]
    xs = [inputs[0], inputs[1], inputs[0], inputs[1]]
    q.route_reset()
    outs = q.qmv_q4_0_q8_1_fused_group(ws, xs)
    singles = [q.qmv_q4_0_q8_1_fused(w, x) for w, x in zip(ws, xs)]
    for a, b in zip(outs, singles):
        assert torch.equal(a, b)
    rc = q.route_counts()
    want = "q4_0_mma_fused_quantize" if q4_kernel == "mma" else "q4_0_stream_fused_quantize"
    assert rc[want] == 5, rc
    for i in (1, 3):
        xq_ref = oracle.quantize_q8_1(xs[i].cpu().numpy())
        y_ref, bound = oracle.q4_0_q8_1(ws[i].cpu().numpy(), xq_ref, K)
        assert_close(f"group[{i}]", outs[i].cpu().numpy(), y_ref, bound)


@pytest.mark.parametrize("M", [1, 3, 8])
def test_q4_0_group_on_q8_1_matches_single_calls(q, q4_kernel, M):
    """The grouped launch on Q8_1 activations is bit-identical to one call per matrix."""
    from gemm_qmv_quantize_gb300 import synth
    K = 4096
    Ns = [4096, 1000, 16]
    ws = [synth.q4_0_weights(n, K, seed=2900 + i, device=DEV) for i, n in enumerate(Ns)]
    xq = [q.qmv_quantize_q8_1(synth.activations_f32(M, K, seed=2990 + j, device=DEV)) for j in range(2)]
    xqs = [xq[0], xq[1], xq[0]]
    outs = q.qmv_q4_0_q8_1_group(ws, xqs, K)
    for w, x, o in zip(ws, xqs, outs):
        assert torch.equal(o, q.qmv_q4_0_q8_1(w, x, K))
    y_ref, bound = oracle.q4_0_q8_1(ws[1].cpu().numpy(), xqs[1].cpu().numpy(), K)
    assert_close("group[1]", outs[1].cpu().numpy(), y_ref, bound)


# ---------------------------------------------------------------- largest K

def test_large_k_routes_and_parity(q):
    """K = 65536: the streaming kernel at M = 1; at M = 8 the staged activations of
    the streaming and tensor-core kernels exceed shared memory, so the single call
    takes the generic kernel and the fused call refuses with QMV_ERR_SHAPE."""
    synth = _synth()
    K, N = 65536, 40
    w = synth.q4_0_weights(N, K, seed=77, device=DEV)
    for M, route in ((1, "q4_0_stream_dp4a"), (8, "q4_0_generic")):
        x = synth.activations_f32(M, K, seed=78 + M, device=DEV)
        xq = q.qmv_quantize_q8_1(x)
        q.route_reset()
        y = q.qmv_q4_0_q8_1(w, xq, K)
        assert q.route_counts()[route] == 1
        y_ref, bound = oracle.q4_0_q8_1(w.cpu().numpy(), xq.cpu().numpy(), K)
        assert_close(f"K=65536 M={M}", y.cpu().numpy(), y_ref, bound)
    from gemm_qmv_quantize_gb300 import QmvError
    with pytest.raises(QmvError, match="QMV_ERR_SHAPE"):
        q.qmv_q4_0_q8_1_fused(w, synth.activations_f32(8, K, seed=90, device=DEV))


# ---------------------------------------------------------------- lane pairs sharing activation records

@pytest.mark.parametrize("M", [2, 3, 4])
@pytest.mark.parametrize("fused", [False, True])
def test_q4_0_lane_pairs_bit_identical(q, monkeypatch, M, fused):
    """K = 4096, enough rows that warps see whole two-row chunks (and an odd last row):
    the lane-pair path gives every output bit-identical to the path that reads all M
    records per lane (the same per-unit arithmetic), and within the bound."""
    synth = _synth()
    N, K = 16 * 1216 + 37, 4096
    w = synth.q4_0_weights(N, K, seed=500 + M, device=DEV)
    x = synth.activations_f32(M, K, seed=510 + M, device=DEV)
    xq = q.qmv_quantize_q8_1(x)
    run = (lambda: q.qmv_q4_0_q8_1_fused(w, x)) if fused else (lambda: q.qmv_q4_0_q8_1(w, xq, K))
    monkeypatch.setenv("QMV_Q4_ACT_REGS_M2", "0")   # M = 2 through the pairs too
    monkeypatch.setenv("QMV_Q4_MMA_MIN_M", "9")
    ys = []
    for pair in ("1", "0"):   # forced on at M = 2..3 too
        monkeypatch.setenv("QMV_Q4_PAIR", pair)
        ys.append(run())
    assert torch.equal(ys[0], ys[1])
    rows = synth.sample_rows(N, 48, seed=M).numpy()
    y_ref, bound = oracle.q4_0_q8_1(np.ascontiguousarray(w.cpu().numpy()[rows]), xq.cpu().numpy(), K)
    assert_close(f"lane pairs M={M}", ys[0].cpu().numpy()[:, rows], y_ref, bound)


@pytest.mark.parametrize("fused", [False, True])
def test_q4_0_m3_register_records_bit_identical(q, monkeypatch, fused):
    """M = 3, K = 4096 with two of the three activation records in registers: every
    output bit-identical to the all-shared-memory path, and within the bound."""
    synth = _synth()
    M, N, K = 3, 16 * 1216 + 37, 4096
    w = synth.q4_0_weights(N, K, seed=530, device=DEV)
    x = synth.activations_f32(M, K, seed=531, device=DEV)
    xq = q.qmv_quantize_q8_1(x)
    run = (lambda: q.qmv_q4_0_q8_1_fused(w, x)) if fused else (lambda: q.qmv_q4_0_q8_1(w, xq, K))
    ys = []
    for on in ("1", "0"):
        monkeypatch.setenv("QMV_Q4_ACT_REGS_M3", on)
        ys.append(run())
    assert torch.equal(ys[0], ys[1])
    rows = synth.sample_rows(N, 48, seed=3).numpy()
    y_ref, bound = oracle.q4_0_q8_1(np.ascontiguousarray(w.cpu().numpy()[rows]), xq.cpu().numpy(), K)
    assert_close("M = 3 register records", ys[0].cpu().numpy()[:, rows], y_ref, bound)

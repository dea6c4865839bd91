"""GPU parity: Q4_K x Q8_1 MMVQ through the C ABI vs the CPU oracle (the dp4a
streaming kernel up to M = 4, the int8 tensor-core kernel from M = 5).

- Integer sub-block sums S = sum q * q8 identical (qmv_debug_q4_k_block_dots runs
  the product kernel's device code with the product kernel choice).
- fp32 outputs within |y - y_ref| <= 1e-3 * sum|w*x| + 1e-6, the oracle's y being
  the plain definition sum_k (d sc q - dmin mn) * d8 q8 in fp64.
- The fused entry points bit-identical to quantize + the Q8_1 entry point.
Shapes span several warps' spans with a ragged tail, M = 1..8, grouped launches
sharing an input, and the full-size matrices of the Qwen3-8B-shaped Q4_K stack
(sampled rows).
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


def _synth():
    from gemm_qmv_quantize_gb300 import synth
    return synth


def _case(q, M, N, K, seed, rows=None):
    synth = _synth()
    w = synth.q4_k_weights(N, K, seed=seed, device=DEV)
    x = synth.activations_f32(M, K, seed=seed + 1, device=DEV)
    xq = q.qmv_quantize_q8_1(x)
    y = q.qmv_q4_k_q8_1(w, xq, K)
    torch.cuda.synchronize()
    wn = w.cpu().numpy() if rows is None else w.cpu().numpy()[rows]
    y_ref, bound = oracle.q4_k_q8_1(wn, xq.cpu().numpy(), K)
    got = y.cpu().numpy() if rows is None else y.cpu().numpy()[:, rows]
    assert_close(f"q4_k M={M} N={N} K={K}", got, y_ref, bound)
    return w, x, xq, y


@pytest.mark.parametrize("M", range(1, 9))
def test_block_dots_exact(q, M):
    synth = _synth()
    N, K = 67, 1024
    w = synth.q4_k_weights(N, K, seed=40 + M, device=DEV)
    xq = q.qmv_quantize_q8_1(synth.activations_f32(M, K, seed=50 + M, device=DEV))
    dots = q.qmv_debug_q4_k_block_dots(w, xq, K)
    S = oracle.q4_k_block_dots(w.cpu().numpy(), xq.cpu().numpy(), K)
    assert np.array_equal(dots.cpu().numpy(), S)


@pytest.mark.parametrize("M", range(1, 9))
def test_multi_span_ragged(q, M):
    """dp4a streaming kernel up to M = 4, int8 tensor cores (m16n8k32) from M = 5."""
    q.route_reset()
    _case(q, M, 16 * 152 + 37, 2048, seed=100 + M)
    assert q.route_counts()["q4_k_stream_dp4a" if M <= 4 else "q4_k_mma_m16n8k32"] == 1


@pytest.mark.parametrize("M", [1, 5, 8])
def test_both_kernels_at_every_m(q, monkeypatch, M):
    """The kernel the planner does not pick for this M, forced: within the bound too."""
    synth = _synth()
    N, K = 16 * 40 + 9, 4096
    w = synth.q4_k_weights(N, K, seed=150 + M, device=DEV)
    xq = q.qmv_quantize_q8_1(synth.activations_f32(M, K, seed=160 + M, device=DEV))
    monkeypatch.setenv("QMV_Q4K_MMA_MIN_M", "1" if M < 5 else "9")
    q.route_reset()
    y = q.qmv_q4_k_q8_1(w, xq, K)
    dots = q.qmv_debug_q4_k_block_dots(w, xq, K)
    assert q.route_counts()["q4_k_mma_m16n8k32" if M < 5 else "q4_k_stream_dp4a"] == 2
    assert np.array_equal(dots.cpu().numpy(), oracle.q4_k_block_dots(w.cpu().numpy(), xq.cpu().numpy(), K))
    y_ref, bound = oracle.q4_k_q8_1(w.cpu().numpy(), xq.cpu().numpy(), K)
    assert_close(f"forced kernel M={M}", y.cpu().numpy(), y_ref, bound)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 7, 512), (5, 33, 4096), (8, 100, 12288), (3, 1, 14336)])
def test_shapes(q, M, N, K):
    _case(q, M, N, K, seed=N + K)


@pytest.mark.parametrize("M", [1, 4, 6, 8])
def test_fused_bit_identical(q, M):
    w, x, xq, y = _case(q, M, 1000, 4096, seed=200 + M)
    q.route_reset()
    yf = q.qmv_q4_k_q8_1_fused(w, x)
    assert q.route_counts()["q4_k_stream_fused_quantize" if M <= 4 else "q4_k_mma_fused_quantize"] == 1
    assert torch.equal(yf, y)


@pytest.mark.parametrize("M", [1, 3, 8])
def test_group_matches_oracle_and_single_calls(q, M):
    """q/k/v-like group sharing one input plus a matrix with its own input."""
    synth = _synth()
    K = 4096
    Ns = [4096, 1024, 1024, 300]
    ws = [synth.q4_k_weights(n, K, seed=300 + i, device=DEV) for i, n in enumerate(Ns)]
    xa = synth.activations_f32(M, K, seed=390, device=DEV)
    xb = synth.activations_f32(M, K, seed=391, device=DEV)
    xs = [xa, xa, xa, xb]
    outs = q.qmv_q4_k_q8_1_fused_group(ws, xs)
    xqs = [q.qmv_quantize_q8_1(x) for x in xs]
    outs_q = q.qmv_q4_k_q8_1_group(ws, xqs, K)
    for i, n in enumerate(Ns):
        single = q.qmv_q4_k_q8_1(ws[i], xqs[i], K)
        assert torch.equal(outs[i], single) and torch.equal(outs_q[i], single)
        rows = np.arange(n) if n < 2000 else synth.sample_rows(n, 64, seed=i).numpy()
        y_ref, bound = oracle.q4_k_q8_1(ws[i].cpu().numpy()[rows], xqs[i].cpu().numpy(), K)
        assert_close(f"group[{i}]", outs[i].cpu().numpy()[:, rows], y_ref, bound)


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("N,K", [(4096, 4096), (1024, 4096), (12288, 4096), (4096, 12288), (151936, 4096)])
def test_qwen3_8b_shapes_sampled(q, M, N, K):
    rows = _synth().sample_rows(N, 48, seed=N + K).numpy()
    _case(q, M, N, K, seed=N * 3 + K + M, rows=rows)


def test_outliers_and_zero_blocks(q):
    """Activation blocks of zeros and of large magnitude; a weight row of zero scales."""
    synth = _synth()
    N, K = 40, 2048
    w = synth.q4_k_weights(N, K, seed=7, device=DEV)
    w[3, :] = 0                                    # d = dmin = 0 everywhere: y = 0
    x = synth.activations_f32(4, K, seed=8, device=DEV)
    x[0, :64] = 0.0
    x[1, 32:64] *= 1e4
    xq = q.qmv_quantize_q8_1(x)
    y = q.qmv_q4_k_q8_1(w, xq, K)
    y_ref, bound = oracle.q4_k_q8_1(w.cpu().numpy(), xq.cpu().numpy(), K)
    assert_close("outliers", y.cpu().numpy(), y_ref, bound)
    assert torch.all(y[:, 3] == 0)


def test_empty_and_k0(q):
    synth = _synth()
    w = synth.q4_k_weights(16, 256, seed=1, device=DEV)
    xq = q.qmv_quantize_q8_1(synth.activations_f32(2, 256, seed=2, device=DEV))
    y = q.qmv_q4_k_q8_1(w[:0], xq, 256)
    assert y.shape == (2, 0)
    out = torch.full((2, 5), 7.0, device=DEV)
    q.lib().qmv_q4_k_q8_1(0, 0, out.data_ptr(), 2, 5, 0, None)   # K = 0: y = 0
    torch.cuda.synchronize()
    assert torch.all(out == 0)

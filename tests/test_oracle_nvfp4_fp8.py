"""Pins of the oracle's NVFP4 W4A16 and FP8 W8A16 skinny GEMM.

- Hand-derived rows (tests/golden/nvfp4_fp8_dot.json).
- fp64 brute force on tiny non-square inputs, with every code decoded by a
  library routine (torch float8_e4m3fn for E4M3) or by the closed form
  (E2M1) and the product taken by numpy: catches a swapped nibble order, a
  scale indexed per 8 or per 32 instead of per 16, a transposed operand.
- Special cases: g = 0, a zero scale group or a zero row scale give zero
  rows; codes of 1.0 with unit scales give y = sum_k x (closed form); a single
  nonzero weight gives w * x exactly; flipping every sign bit negates y.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import GOLDEN

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def _e4m3(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _rand_nvfp4(rng, N, K):
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    s = torch.from_numpy(np.abs(rng.standard_normal((N, K // 16))) * 0.5)
    scales = s.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scales


def _dequant_nvfp4(codes, scales, g):
    N = codes.shape[0]
    c = np.stack([codes & 0x0F, codes >> 4], axis=2).reshape(N, -1)   # k even low, k odd high
    s = np.repeat(_e4m3(scales), 16, axis=1)
    return E2M1[c] * s * np.float64(np.float32(g))


def test_golden_rows():
    with open(os.path.join(GOLDEN, "nvfp4_fp8_dot.json")) as f:
        g = json.load(f)
    a = g["nvfp4"]
    y, _ = oracle.nvfp4_w4a16(np.array([a["codes"]], np.uint8), np.array([[a["scale"]]], np.uint8),
                              a["g"], np.array([a["x"]], np.float16))
    assert y[0, 0] == a["y"]
    b = g["fp8"]
    y, _ = oracle.fp8_w8a16(np.array([b["w"]], np.uint8), np.array([b["row_scale"]], np.float32),
                            np.array([b["x"]], np.float16))
    assert y[0, 0] == b["y"]


@pytest.mark.parametrize("M,N,K", [(1, 3, 16), (2, 5, 48), (5, 4, 128), (8, 3, 256)])
def test_nvfp4_brute_force(M, N, K):
    rng = np.random.default_rng(M + 10 * N + K)
    codes, scales = _rand_nvfp4(rng, N, K)
    x = rng.standard_normal((M, K)).astype(np.float16)
    g = 0.01
    y, bound = oracle.nvfp4_w4a16(codes, scales, g, x)
    W = _dequant_nvfp4(codes, scales, g)
    X = x.astype(np.float64)
    assert np.allclose(y, X @ W.T, rtol=1e-12, atol=1e-14)
    assert np.allclose(bound, np.abs(X) @ np.abs(W).T, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("M,N,K", [(1, 3, 8), (3, 4, 40), (8, 5, 128)])
def test_fp8_brute_force(M, N, K):
    rng = np.random.default_rng(M + 10 * N + K)
    w = torch.from_numpy(rng.standard_normal((N, K))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    rs = (np.abs(rng.standard_normal(N)) + 0.01).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float16)
    y, bound = oracle.fp8_w8a16(w, rs, x)
    W = _e4m3(w) * rs.astype(np.float64)[:, None]
    X = x.astype(np.float64)
    assert np.allclose(y, X @ W.T, rtol=1e-12, atol=1e-14)
    assert np.allclose(bound, np.abs(X) @ np.abs(W).T, rtol=1e-12, atol=1e-14)


def test_nvfp4_special_cases():
    rng = np.random.default_rng(21)
    M, N, K = 3, 4, 64
    codes, scales = _rand_nvfp4(rng, N, K)
    x = rng.standard_normal((M, K)).astype(np.float16)
    y, _ = oracle.nvfp4_w4a16(codes, scales, 0.0, x)
    assert np.all(y == 0.0)
    zs = scales.copy()
    zs[1, :] = 0
    y, _ = oracle.nvfp4_w4a16(codes, zs, 0.01, x)
    assert np.all(y[:, 1] == 0.0) and np.any(y[:, 0] != 0.0)
    # every code 1.0 (0x2 in both nibbles), scale 1.0 (0x38), g = 1 -> y = sum_k x
    ones = np.full((N, K // 2), 0x22, np.uint8)
    unit = np.full((N, K // 16), 0x38, np.uint8)
    y, _ = oracle.nvfp4_w4a16(ones, unit, 1.0, x)
    assert np.allclose(y, np.repeat(x.astype(np.float64).sum(axis=1, keepdims=True), N, axis=1), rtol=1e-14)
    # single nonzero weight: code 0x7 (6.0) at k = 37 of row 2, scale 0x40 (2.0), g = 0.5
    single = np.zeros((N, K // 2), np.uint8)
    single[2, 37 // 2] = 0x7 << 4          # k odd -> high nibble
    s2 = np.full((N, K // 16), 0x40, np.uint8)
    y, _ = oracle.nvfp4_w4a16(single, s2, 0.5, x)
    assert np.array_equal(y[:, 2], 6.0 * 2.0 * 0.5 * x[:, 37].astype(np.float64))
    assert np.all(y[:, [0, 1, 3]] == 0.0)
    # flipping every sign bit negates the result
    y1, _ = oracle.nvfp4_w4a16(codes, scales, 0.01, x)
    y2, _ = oracle.nvfp4_w4a16(codes ^ 0x88, scales, 0.01, x)
    assert np.array_equal(y2, -y1)


def test_fp8_special_cases():
    rng = np.random.default_rng(23)
    M, N, K = 2, 3, 32
    w = torch.from_numpy(rng.standard_normal((N, K))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    x = rng.standard_normal((M, K)).astype(np.float16)
    rs = np.array([0.02, 0.0, 0.5], np.float32)
    y, _ = oracle.fp8_w8a16(w, rs, x)
    assert np.all(y[:, 1] == 0.0)
    ones = np.full((N, K), 0x38, np.uint8)
    y, _ = oracle.fp8_w8a16(ones, np.ones(N, np.float32), x)
    assert np.allclose(y, np.repeat(x.astype(np.float64).sum(axis=1, keepdims=True), N, axis=1), rtol=1e-14)
    y1, _ = oracle.fp8_w8a16(w, rs, x)
    y2, _ = oracle.fp8_w8a16(w ^ 0x80, rs, x)
    assert np.array_equal(y2, -y1)


def test_fp16_outliers_stay_finite():
    """Activation outliers at the top of the fp16 range (the overflow case of
    'v100-skinny README', section 'How QPN works') stay exact in fp64."""
    rng = np.random.default_rng(29)
    N, K = 3, 64
    codes, scales = _rand_nvfp4(rng, N, K)
    x = rng.standard_normal((1, K)).astype(np.float16)
    x[0, 5] = np.float16(60000.0)
    x[0, 9] = np.float16(-65504.0)
    y, bound = oracle.nvfp4_w4a16(codes, scales, 0.01, x)
    W = _dequant_nvfp4(codes, scales, 0.01)
    assert np.all(np.isfinite(y))
    assert np.allclose(y, x.astype(np.float64) @ W.T, rtol=1e-12)

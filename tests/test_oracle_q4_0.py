"""Pins of the oracle's Q4_0 x Q8_1 mat-vec.

- The hand-derived block of tests/golden/q4_0_dot.json.
- fp64 brute force on tiny non-square inputs: the weights and activations are
  dequantized with numpy (float16 view for the scales, bit masks for the
  nibbles) and multiplied with a matrix product, so a swapped nibble half, a
  dropped -8 offset, a transposed operand or a wrong block index fails.
- The offset-8 identity y = sum_b d4 * (d8 * S_b - 8 * s8_b): exact when s8 is
  taken as d8 * T, and within the rounding of the stored fp16 s8 otherwise.
- Special cases: d4 = 0 -> y = 0; every nibble 8 -> y = 0; every nibble 9 ->
  y = sum_b d4 d8 T_b; scaling every d4 by 2 doubles y exactly.
"""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _rand_q4_0(rng, N, K):
    nb = K // 32
    d = (np.abs(rng.standard_normal((N, nb))) * 0.01).astype(np.float16)
    blocks = np.zeros((N, nb, 18), dtype=np.uint8)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:] = rng.integers(0, 256, (N, nb, 16), dtype=np.uint8)
    return blocks.reshape(N, nb * 18)


def _dequant_q4_0(w, K):
    N, nb = w.shape[0], K // 32
    b = w.reshape(N, nb, 18)
    d = b[:, :, 0:2].copy().view(np.float16).astype(np.float64)       # [N, nb, 1]
    qs = b[:, :, 2:]
    q = np.concatenate([qs & 0x0F, qs >> 4], axis=2).astype(np.float64)  # elements 0..15, 16..31
    return (d * (q - 8.0)).reshape(N, K)


def _dequant_q8_1(xq, K):
    M, nb = xq.shape[0], K // 32
    b = xq.reshape(M, nb, 36)
    d = b[:, :, 0:2].copy().view(np.float16).astype(np.float64)
    q = b[:, :, 4:].view(np.int8).astype(np.float64)
    return (d * q).reshape(M, K)


def test_golden_block():
    with open(os.path.join(GOLDEN, "q4_0_dot.json")) as f:
        g = json.load(f)
    with open(os.path.join(GOLDEN, "q8_1_blocks.json")) as f:
        cases = {c["name"]: c for c in json.load(f)["cases"]}
    x = np.array(cases[g["q8_case"]]["x"], dtype=np.float32)[None, :]
    xq = oracle.quantize_q8_1(x)
    d4 = int(g["d4"], 16)
    qs = [(j & 15) | ((15 - j) << 4) for j in range(16)]
    w = np.array([d4 & 0xFF, d4 >> 8] + qs, dtype=np.uint8)[None, :]
    S, T = oracle.q4_0_block_dots(w, xq, 32)
    y, _ = oracle.q4_0_q8_1(w, xq, 32)
    assert S[0, 0, 0] == g["S"] and T[0, 0] == g["T"]
    assert y[0, 0] == g["y"]


@pytest.mark.parametrize("M,N,K", [(1, 3, 32), (2, 5, 64), (3, 7, 96), (8, 4, 256)])
def test_brute_force_tiny(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    w = _rand_q4_0(rng, N, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = oracle.quantize_q8_1(x)
    y, bound = oracle.q4_0_q8_1(w, xq, K)
    W = _dequant_q4_0(w, K)
    X = _dequant_q8_1(xq, K)
    ref = X @ W.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)
    assert np.allclose(bound, np.abs(X) @ np.abs(W).T, rtol=1e-12, atol=1e-15)


def test_block_dots_brute_force():
    rng = np.random.default_rng(3)
    M, N, K = 3, 6, 128
    w = _rand_q4_0(rng, N, K)
    xq = oracle.quantize_q8_1(rng.standard_normal((M, K)).astype(np.float32))
    S, T = oracle.q4_0_block_dots(w, xq, K)
    qs = w.reshape(N, K // 32, 18)[:, :, 2:]
    q4 = np.concatenate([qs & 0x0F, qs >> 4], axis=2).astype(np.int64)        # [N, nb, 32]
    q8 = xq.reshape(M, K // 32, 36)[:, :, 4:].view(np.int8).astype(np.int64)  # [M, nb, 32]
    assert np.array_equal(S, np.einsum("nbj,mbj->mnb", q4, q8))
    assert np.array_equal(T, q8.sum(axis=2))


def test_offset_identity():
    rng = np.random.default_rng(5)
    M, N, K = 2, 9, 256
    w = _rand_q4_0(rng, N, K)
    xq = oracle.quantize_q8_1(rng.standard_normal((M, K)).astype(np.float32))
    y, bound = oracle.q4_0_q8_1(w, xq, K)
    S, T = oracle.q4_0_block_dots(w, xq, K)
    nb = K // 32
    d4 = w.reshape(N, nb, 18)[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    xb = xq.reshape(M, nb, 36)
    d8 = xb[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    s8 = xb[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    # exact form: s8 replaced by d8 * T
    exact = np.einsum("nb,mnb->mn", d4, d8[:, None, :] * S - 8.0 * (d8 * T)[:, None, :])
    assert np.allclose(y, exact, rtol=1e-12, atol=1e-15)
    # stored s8 differs from d8*T by the fp16 roundings of d and d*T (2 half-ulps)
    approx = np.einsum("nb,mnb->mn", d4, d8[:, None, :] * S - 8.0 * s8[:, None, :])
    slack = np.einsum("nb,mb->mn", np.abs(d4), 8.0 * np.abs(d8 * T) * 2.0 ** -10 * 1.01 + 8.0 * 2.0 ** -24)
    assert np.all(np.abs(approx - y) <= slack)


def test_special_cases():
    rng = np.random.default_rng(9)
    M, N, K = 2, 4, 128
    nb = K // 32
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = oracle.quantize_q8_1(x)
    w = _rand_q4_0(rng, N, K)

    zero_scale = w.copy().reshape(N, nb, 18)
    zero_scale[:, :, 0:2] = 0
    y, _ = oracle.q4_0_q8_1(zero_scale.reshape(N, -1), xq, K)
    assert np.all(y == 0.0)

    eights = w.copy().reshape(N, nb, 18)
    eights[:, :, 2:] = 0x88
    y, bound = oracle.q4_0_q8_1(eights.reshape(N, -1), xq, K)
    assert np.all(y == 0.0) and np.all(bound == 0.0)

    nines = w.copy().reshape(N, nb, 18)
    nines[:, :, 2:] = 0x99
    y, _ = oracle.q4_0_q8_1(nines.reshape(N, -1), xq, K)
    _, T = oracle.q4_0_block_dots(nines.reshape(N, -1), xq, K)
    d4 = nines[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    d8 = xq.reshape(M, nb, 36)[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    assert np.allclose(y, (d8 * T) @ d4.T, rtol=1e-12)

    doubled = w.copy().reshape(N, nb, 18)
    d = doubled[:, :, 0:2].copy().view(np.float16)
    doubled[:, :, 0:2] = (d * np.float16(2)).view(np.uint8)
    y1, _ = oracle.q4_0_q8_1(w, xq, K)
    y2, _ = oracle.q4_0_q8_1(doubled.reshape(N, -1), xq, K)
    assert np.array_equal(y2, 2.0 * y1)


def test_constant_activation_closed_form():
    """x = c everywhere -> every q8 = 127 and d8 = fp16(c/127): y = d8*127*sum(d4*(q4-8))."""
    rng = np.random.default_rng(13)
    N, K = 3, 64
    w = _rand_q4_0(rng, N, K)
    c = np.float32(0.75)
    xq = oracle.quantize_q8_1(np.full((1, K), c, dtype=np.float32))
    assert np.all(xq.reshape(-1, 36)[:, 4:].view(np.int8) == 127)
    d8 = float(np.float16(c / np.float32(127)))
    W = _dequant_q4_0(w, K)
    y, _ = oracle.q4_0_q8_1(w, xq, K)
    assert np.allclose(y[0], d8 * 127.0 * W.sum(axis=1), rtol=1e-12)

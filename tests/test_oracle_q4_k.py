"""Pins of the oracle's Q4_K x Q8_1 mat-vec (llama.cpp's K-quant super-block; the
pages name the Q4_K_M models in "Machine Learning on NVIDIA CMP", section
"llama.cpp results", without printing the layout).

- Hand-derived unpacking of the 12 packed 6-bit scale / minimum bytes, and a
  round trip through a packer written here in the opposite direction.
- Hand-derived element positions: element 64c + e is the low nibble of data
  byte 32c + e, element 64c + 32 + e its high nibble.
- The Q4_0 identity: with dmin = d and every minimum 8x its scale, a Q4_K
  super-block is eight Q4_0 blocks with d4 = d * sc (w = d sc (q - 8)); the
  oracle must agree with its (separately pinned) Q4_0 routine on the same
  nibbles, integer block dots bit-exact and outputs to fp64 rounding.
- Closed forms: zero scales and minimums give y = 0; all nibbles 0 give
  y = -dmin * sum_j mn_j * sum_{k in j} xhat_k; positive weights and
  activations give bound == y.
"""
import numpy as np
import pytest

import oracle

D_ONE = np.float16(1.0)


def _pack_scales(sc, mn):
    """The 12 packed bytes of eight 6-bit (scale, minimum) pairs: the low 6 bits
    of sub-blocks 0..3 in bytes 0..3 (scales) and 4..7 (minimums); sub-blocks
    4..7 keep their low 4 bits in bytes 8..11 (scale low, minimum high nibble)
    and their top 2 bits in the top 2 bits of bytes 0..3 (scales) and 4..7
    (minimums)."""
    p = np.zeros(12, dtype=np.uint8)
    for j in range(4):
        p[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        p[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        p[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return p


def _superblock(d, dmin, sc, mn, q):
    """One 144-byte super-block from fp16 d, dmin, eight (sc, mn) and 256 nibbles
    q[i] (element i), placed as the format says."""
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    b[2:4] = np.array([dmin], dtype=np.float16).view(np.uint8)
    b[4:16] = _pack_scales(sc, mn)
    for c in range(4):
        for e in range(32):
            b[16 + 32 * c + e] = (q[64 * c + e] & 15) | ((q[64 * c + 32 + e] & 15) << 4)
    return b


def _q8_1_rows(rng, M, K):
    return oracle.quantize_q8_1(rng.standard_normal((M, K)).astype(np.float32))


def _xhat(xq, K):
    """Dequantized Q8_1 activations d8 * q8 (numpy float16 view of d8)."""
    M, nb = xq.shape[0], K // 32
    b = xq.reshape(M, nb, 36)
    d8 = b[:, :, 0:2].copy().view(np.float16).astype(np.float64)
    q8 = b[:, :, 4:].view(np.int8).astype(np.float64)
    return (d8 * q8).reshape(M, K)


def test_scale_min_hand_derived():
    # bytes 0, 21, 42, ..., 231 (21 i); values worked out by hand from the layout
    p = (np.arange(12) * 21).astype(np.uint8)
    expect = [(0, 20), (21, 41), (42, 62), (63, 19), (8, 26), (13, 27), (2, 29), (7, 46)]
    assert [oracle.q4_k_scale_min(p, j) for j in range(8)] == expect


def test_scale_min_round_trip():
    rng = np.random.default_rng(5)
    for _ in range(200):
        sc = rng.integers(0, 64, 8)
        mn = rng.integers(0, 64, 8)
        p = _pack_scales(sc, mn)
        assert [oracle.q4_k_scale_min(p, j) for j in range(8)] == list(zip(sc.tolist(), mn.tolist()))


def test_element_positions_hand_derived():
    # d = 1, dmin = 0, every scale 1: each weight is its nibble. Byte 32c + e of the
    # data holds element 64c + e (low nibble) and 64c + 32 + e (high nibble).
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.array([D_ONE], dtype=np.float16).view(np.uint8)
    b[4:16] = _pack_scales([1] * 8, [0] * 8)
    b[16 + 0] = 0x21      # element 0 = 1, element 32 = 2
    b[16 + 31] = 0x43     # element 31 = 3, element 63 = 4
    b[16 + 32] = 0x65     # element 64 = 5, element 96 = 6
    b[16 + 127] = 0xF7    # element 223 = 7, element 255 = 15
    w = oracle.q4_k_dequantize(b[None, :], 256)[0]
    expect = np.zeros(256)
    expect[[0, 32, 31, 63, 64, 96, 223, 255]] = [1, 2, 3, 4, 5, 6, 7, 15]
    assert np.array_equal(w, expect)


def test_minimum_subtracted_per_sub_block():
    # all nibbles 0: w = -dmin * mn[j] on sub-block j; dmin differs from d
    mn = [1, 2, 3, 4, 5, 6, 7, 63]
    b = _superblock(np.float16(0.5), np.float16(0.25), [9] * 8, mn, np.zeros(256, dtype=np.int64))
    w = oracle.q4_k_dequantize(b[None, :], 256)[0]
    assert np.array_equal(w, np.repeat(-0.25 * np.array(mn, dtype=np.float64), 32))


def _q4_0_from_nibbles(q, d4):
    """Q4_0 blocks [nb][18] from logical nibbles q[k] and block scales d4[b]:
    element j of a block in the low nibble of byte j (j < 16), else the high
    nibble of byte j - 16."""
    nb = len(q) // 32
    out = np.zeros((nb, 18), dtype=np.uint8)
    for bi in range(nb):
        out[bi, 0:2] = np.array([d4[bi]], dtype=np.float16).view(np.uint8)
        blk = q[32 * bi:32 * bi + 32]
        out[bi, 2:] = (blk[:16] & 15) | ((blk[16:] & 15) << 4)
    return out.reshape(-1)


@pytest.mark.parametrize("M,N,K", [(1, 3, 256), (3, 5, 512), (2, 4, 1024)])
def test_q4_0_identity(M, N, K):
    """dmin = d, mn = 8 sc (sc <= 7) and d a power of two: Q4_K == Q4_0 with d4 = d sc."""
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    nsb = K // 256
    q = rng.integers(0, 16, (N, K))
    wk = np.zeros((N, nsb * 144), dtype=np.uint8)
    w0 = np.zeros((N, K // 32 * 18), dtype=np.uint8)
    for n in range(N):
        d4 = []
        for s in range(nsb):
            d = np.float16(2.0 ** -int(rng.integers(4, 10)))
            sc = rng.integers(0, 8, 8)
            wk[n, s * 144:(s + 1) * 144] = _superblock(d, d, sc, 8 * sc, q[n, 256 * s:256 * (s + 1)])
            d4 += [np.float16(float(d) * int(c)) for c in sc]   # exact: sc <= 7
        w0[n] = _q4_0_from_nibbles(q[n], d4)
    xq = _q8_1_rows(rng, M, K)
    S4k = oracle.q4_k_block_dots(wk, xq, K)
    S40, _ = oracle.q4_0_block_dots(w0, xq, K)
    assert np.array_equal(S4k, S40)
    yk, bk = oracle.q4_k_q8_1(wk, xq, K)
    y0, b0 = oracle.q4_0_q8_1(w0, xq, K)
    assert np.allclose(yk, y0, rtol=1e-12, atol=1e-12)
    assert np.allclose(bk, b0, rtol=1e-12, atol=1e-12)


def test_block_dots_brute_force():
    """S = sum over each 32-block of nibble * q8, from the logical nibbles."""
    rng = np.random.default_rng(17)
    N, K, M = 3, 512, 2
    q = rng.integers(0, 16, (N, K))
    w = np.stack([np.concatenate([_superblock(np.float16(0.01), np.float16(0.02), rng.integers(0, 64, 8),
                                              rng.integers(0, 64, 8), q[n, 256 * s:256 * (s + 1)])
                                  for s in range(K // 256)]) for n in range(N)])
    xq = _q8_1_rows(rng, M, K)
    q8 = xq.reshape(M, K // 32, 36)[:, :, 4:].view(np.int8).astype(np.int64).reshape(M, K)
    expect = np.einsum("nbi,mbi->mnb", q.reshape(N, K // 32, 32), q8.reshape(M, K // 32, 32))
    assert np.array_equal(oracle.q4_k_block_dots(w, xq, K), expect)


def test_zero_scales_and_minimums():
    rng = np.random.default_rng(3)
    K = 512
    w = np.concatenate([_superblock(np.float16(0.3), np.float16(0.7), [0] * 8, [0] * 8,
                                    rng.integers(0, 16, 256)) for _ in range(2)])[None, :]
    y, bound = oracle.q4_k_q8_1(w, _q8_1_rows(rng, 2, K), K)
    assert np.all(y == 0) and np.all(bound == 0)


def test_all_zero_nibbles_closed_form():
    rng = np.random.default_rng(4)
    K = 512
    mn = [rng.integers(0, 64, 8) for _ in range(2)]
    w = np.concatenate([_superblock(np.float16(0.5), np.float16(0.125), rng.integers(0, 64, 8), mn[s],
                                    np.zeros(256, dtype=np.int64)) for s in range(2)])[None, :]
    xq = _q8_1_rows(rng, 3, K)
    xh = _xhat(xq, K).reshape(3, K // 32, 32).sum(axis=2)                 # [M][16 sub-blocks]
    expect = -0.125 * (xh * np.concatenate(mn).astype(np.float64)).sum(axis=1)
    y, _ = oracle.q4_k_q8_1(w, xq, K)
    assert np.allclose(y[:, 0], expect, rtol=1e-12, atol=1e-15)


def test_positive_bound_equals_y():
    """Positive weights (minimums 0, nibbles >= 1) against positive activations."""
    rng = np.random.default_rng(6)
    K = 256
    w = _superblock(np.float16(0.01), np.float16(0.5), rng.integers(1, 64, 8), [0] * 8,
                    rng.integers(1, 16, 256))[None, :]
    xq = oracle.quantize_q8_1(np.abs(rng.standard_normal((2, K))).astype(np.float32) + 0.1)
    y, bound = oracle.q4_k_q8_1(w, xq, K)
    assert np.all(y > 0) and np.allclose(y, bound, rtol=1e-13)

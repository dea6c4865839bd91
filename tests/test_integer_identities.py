"""Arithmetic identities behind the kernels, checked on the CPU with a plain
emulation of the instructions (PTX ISA semantics, IEEE fp32) against the oracle:
the exact block sums S = sum q4u * q8 and T = sum q8, the Q4_K scale decode, and
the Q8_1 bytes.

- "Machine Learning on NVIDIA CMP", section "The DP2A patch", rests on splitting a
  4-way int8 dot into two 2-way dots: with A's four bytes sign-extended to int16
  pairs (bytes 0, 1 in one word, bytes 2, 3 in the other), the 2-way dot of the
  first word with B's bytes 0..1 plus that of the second with B's bytes 2..3 is the
  4-way dot, for every A and B (plain algebra: the sum over four products regrouped).
- The dp4a streaming kernel: unsigned low nibbles (mask 0x0f) and high nibbles kept
  in place (mask 0xf0, i.e. 16 q) against signed Q8_1 bytes, so S = lo + hi / 16
  exactly, and a block's dot is S - 8 T.
- The int8 tensor-core kernel: the weight bytes 16 (q - 8) as int8, formed as
  (nibble << 4) ^ 0x80, so a block's product is 16 (S - 8 T) exactly in int32.
- The tensor-core kernel's m16n8k32 fragments: rebuilt into A and B by the PTX
  layout, their product lands 16 (S - 8T) in the lanes the epilogue reads.
- The Q4_0 unit layout: the 36 aligned words of a 144-byte unit give each block's
  scale and nibble words (even blocks realigned by one byte permute).
- The Q8_1 quantizer: x * fl(1 / d) rounded to nearest, redone with the IEEE
  quotient and ties away from zero only near a half-integer, gives the oracle's
  bytes (random, wide-range, subnormal-scale and one-ulp-from-a-tie blocks).
"""
import numpy as np
import pytest

import oracle


def _u8(w):
    w = np.asarray(w, dtype=np.uint32)
    return [((w >> (8 * i)) & 0xFF).astype(np.int64) for i in range(4)]


def _s8(w):
    return [np.where(b >= 128, b - 256, b) for b in _u8(w)]


def dp4a(a, b, c, a_signed=True):
    """dp4a.{s32|u32}.s32: c + sum_i a.byte[i] * b.byte[i], b signed."""
    av = _s8(a) if a_signed else _u8(a)
    bv = _s8(b)
    return c + sum(x * y for x, y in zip(av, bv))


def prmt(a, b, sel):
    """prmt.b32 default mode: result byte i = byte (sel nibble i & 7) of {b, a}
    (a = bytes 0..3, b = bytes 4..7), or that byte's sign bit replicated when the
    nibble's bit 3 is set."""
    src = _u8(a) + _u8(b)
    out = np.zeros_like(np.asarray(a, dtype=np.int64))
    for i in range(4):
        nib = (sel >> (4 * i)) & 0xF
        byte = src[nib & 7]
        if nib & 8:
            byte = np.where(byte & 0x80, 0xFF, 0x00)
        out |= byte << (8 * i)
    return out


def dp2a(a, b, c, hi):
    """dp2a.{lo|hi}.s32.s32: c + a.half[0] * b.byte[o] + a.half[1] * b.byte[o + 1],
    o = 2 for .hi, 0 for .lo; a as two int16, b as four int8."""
    a = np.asarray(a, dtype=np.int64)
    h0, h1 = a & 0xFFFF, (a >> 16) & 0xFFFF
    h0, h1 = np.where(h0 >= 1 << 15, h0 - (1 << 16), h0), np.where(h1 >= 1 << 15, h1 - (1 << 16), h1)
    bv = _s8(b)
    o = 2 if hi else 0
    return c + h0 * bv[o] + h1 * bv[o + 1]


def _int16_pair(lo, hi):
    """Two signed values packed as int16 halves of a 32-bit word (lo in bits 0..15)."""
    return (np.asarray(lo, dtype=np.int64) & 0xFFFF) | ((np.asarray(hi, dtype=np.int64) & 0xFFFF) << 16)


def test_dp4a_equals_two_dp2a_over_sign_extended_halves():
    rng = np.random.default_rng(11)
    edges = np.array([0, 0x7F7F7F7F, 0x80808080, 0xFFFFFFFF, 0x017F80FF, 0x80FF017F], dtype=np.uint64)
    a = np.concatenate([rng.integers(0, 1 << 32, 200_000, dtype=np.uint64), np.repeat(edges, len(edges))])
    b = np.concatenate([rng.integers(0, 1 << 32, 200_000, dtype=np.uint64), np.tile(edges, len(edges))])
    c = rng.integers(-(1 << 20), 1 << 20, len(a))
    a0, a1, a2, a3 = _s8(a)   # A's bytes as signed values, sign-extended by the arithmetic itself
    ref = dp4a(a, b, c)
    assert np.array_equal(dp2a(_int16_pair(a2, a3), b, dp2a(_int16_pair(a0, a1), b, c, hi=False), hi=True), ref)
    # the split is exact only with sign extension: zero-extended halves miss 256 per negative byte
    zext = dp2a(_int16_pair(a2 & 0xFF, a3 & 0xFF), b, dp2a(_int16_pair(a0 & 0xFF, a1 & 0xFF), b, c, hi=False),
                hi=True)
    assert not np.array_equal(zext, ref)


def _blocks(seed, N=37, M=3, K=1024):
    from gemm_qmv_quantize_gb300 import synth
    w = synth.q4_0_weights(N, K, seed=seed).numpy()
    xq = oracle.quantize_q8_1(synth.activations_f32(M, K, seed=seed + 1).numpy())
    # extreme activation blocks: all +127 and all -127 quants
    xq[0, 4:36] = 127
    xq[1, 40:72] = np.uint8(129)   # -127
    S, T = oracle.q4_0_block_dots(w, xq, K)
    nb = K // 32
    qs = w.reshape(N, nb, 18)[:, :, 2:].copy().view("<u4")     # [N][nb][4] words of nibbles
    q8 = xq.reshape(M, nb, 36)[:, :, 4:].copy().view("<u4")    # [M][nb][8] words of int8
    return qs.astype(np.uint64), q8.astype(np.uint64), S.astype(np.int64), T.astype(np.int64)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_stream_kernel_block_dot(seed):
    qs, q8, S, T = _blocks(seed)
    lo = sum(dp4a(qs[None, :, :, i] & 0x0F0F0F0F, q8[:, None, :, i], 0, a_signed=False) for i in range(4))
    hi = sum(dp4a(qs[None, :, :, i] & 0xF0F0F0F0, q8[:, None, :, 4 + i], 0, a_signed=False) for i in range(4))
    assert np.all(hi % 16 == 0)                       # the kept-in-place high nibbles are 16 q
    assert np.array_equal(lo + (hi >> 4), S)          # arithmetic shift: exact on multiples of 16
    assert np.array_equal(lo + (hi >> 4) - 8 * T[:, None, :], S - 8 * T[:, None, :])


@pytest.mark.parametrize("seed", [4, 5])
def test_tensor_core_kernel_bytes(seed):
    qs, q8, S, T = _blocks(seed)
    f_lo = ((qs << 4) & 0xF0F0F0F0) ^ 0x80808080      # int8 bytes 16 (q_lo - 8)
    f_hi = (qs & 0xF0F0F0F0) ^ 0x80808080             # int8 bytes 16 (q_hi - 8)
    for i in range(4):                                # byte 0 of each word: its low nibble q
        q = (qs[..., i] & 0xF).astype(np.int64)
        assert np.array_equal(_s8(f_lo[..., i])[0], 16 * (q - 8))
    D = sum(dp4a(f_lo[None, :, :, i], q8[:, None, :, i], 0) + dp4a(f_hi[None, :, :, i], q8[:, None, :, 4 + i], 0)
            for i in range(4))
    assert np.array_equal(D, 16 * (S - 8 * T[:, None, :]))
    assert np.abs(D).max() < 1 << 31                  # fits the int32 accumulator


def test_q4_k_word_wide_scale_unpack():
    """The Q4_K streaming kernel unpacks the 12 packed bytes with four word-wide
    mask/shift pairs (w1 = bytes 0..3, w2 = 4..7, w3 = 8..11): byte j of
    w1 & 0x3f3f3f3f / w2 & 0x3f3f3f3f are scale / minimum of sub-block j < 4, byte j of
    (w3 & 0x0f0f0f0f) | ((w1 >> 2) & 0x30303030) and
    ((w3 >> 4) & 0x0f0f0f0f) | ((w2 >> 2) & 0x30303030) those of sub-block 4 + j."""
    rng = np.random.default_rng(21)
    packs = np.concatenate([rng.integers(0, 256, (3000, 12), dtype=np.uint8),
                            np.full((1, 12), 0xFF, np.uint8), np.zeros((1, 12), np.uint8)])
    for p in packs:
        w1, w2, w3 = (int(v) for v in p.view("<u4"))
        words = {"sc_lo": w1 & 0x3F3F3F3F, "mn_lo": w2 & 0x3F3F3F3F,
                 "sc_hi": (w3 & 0x0F0F0F0F) | ((w1 >> 2) & 0x30303030),
                 "mn_hi": ((w3 >> 4) & 0x0F0F0F0F) | ((w2 >> 2) & 0x30303030)}
        for j in range(4):
            assert oracle.q4_k_scale_min(p, j) == ((words["sc_lo"] >> 8 * j) & 0xFF, (words["mn_lo"] >> 8 * j) & 0xFF)
            assert oracle.q4_k_scale_min(p, 4 + j) == ((words["sc_hi"] >> 8 * j) & 0xFF,
                                                       (words["mn_hi"] >> 8 * j) & 0xFF)


@pytest.mark.parametrize("seed", [6, 7])
def test_q4_k_stream_sub_block_dots(seed):
    """Data words 8c .. 8c + 7 of a super-block hold sub-block 2c in their low nibbles
    and 2c + 1 in their high nibbles: low nibbles (mask 0x0f) against activation block
    2c, high nibbles in place (mask 0xf0, 16 q) against block 2c + 1, exactly S."""
    from gemm_qmv_quantize_gb300 import synth
    N, M, K = 29, 2, 1024
    w = synth.q4_k_weights(N, K, seed=seed).numpy()
    xq = oracle.quantize_q8_1(synth.activations_f32(M, K, seed=seed + 1).numpy())
    xq[1, 4:36] = np.uint8(129)   # a block of -127 quants
    S = oracle.q4_k_block_dots(w, xq, K).astype(np.int64)
    nsb, nb = K // 256, K // 32
    data = w.reshape(N, nsb, 144)[:, :, 16:].copy().view("<u4").astype(np.uint64)   # [N][nsb][32] words
    q8 = xq.reshape(M, nb, 36)[:, :, 4:].copy().view("<u4").astype(np.uint64)       # [M][nb][8] words
    for s in range(nsb):
        for c in range(4):
            b_lo, b_hi = 8 * s + 2 * c, 8 * s + 2 * c + 1
            lo = sum(dp4a(data[None, :, s, 8 * c + i] & 0x0F0F0F0F, q8[:, None, b_lo, i], 0, a_signed=False)
                     for i in range(8))
            hi = sum(dp4a(data[None, :, s, 8 * c + i] & 0xF0F0F0F0, q8[:, None, b_hi, i], 0, a_signed=False)
                     for i in range(8))
            assert np.all(hi % 16 == 0)
            assert np.array_equal(lo, S[:, :, b_lo]) and np.array_equal(hi >> 4, S[:, :, b_hi])


def _q8_fast_path(x):
    """The device quantizer's per-block arithmetic in IEEE fp32 (numpy rounds like
    the device's non-fast-math ops): d = amax / 127; t = x * fl(1 / d) rounded to
    nearest even; where t lies within 2^-13 of a half-integer, or 1 / d overflows, the
    value is redone as roundf(x / d) (ties away from zero) with the IEEE quotient."""
    x = x.astype(np.float32)
    amax = np.abs(x).max(axis=1)
    d = (amax / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        inv = (np.float32(1) / d).astype(np.float32)
    rcp = np.where(d == 0, np.float32(0), inv).astype(np.float32)
    t = (x * rcp[:, None]).astype(np.float32)
    n = np.rint(t)
    with np.errstate(invalid="ignore"):   # t = inf where 1 / d overflowed: redone below
        slow = np.abs(t - n) > np.float32(0.5 - 2.0 ** -13)
    slow |= (~np.isfinite(inv) & (d != 0))[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        qd = (x / d[:, None]).astype(np.float32)
    away = np.sign(qd) * np.floor(np.abs(qd.astype(np.float64)) + 0.5)
    q = np.where(slow, np.clip(away, -127, 127), n)
    return np.where(d[:, None] == 0, 0, q).astype(np.int64)


def test_quantizer_fast_path_matches_the_oracle():
    rng = np.random.default_rng(31)
    blocks = [rng.standard_normal((20000, 32)),
              rng.standard_normal((2000, 32)) * 1e-40,                      # subnormal amax: 1 / d overflows
              np.exp(rng.uniform(-80, 80, (2000, 32))) * rng.choice([-1, 1], (2000, 32))]
    # adversarial: every value near a tie of x / d, for random scales
    d = np.exp(rng.uniform(-20, 20, 4000)).astype(np.float32)
    k = rng.integers(-126, 127, (4000, 31)) + 0.5
    near = (k * d[:, None]).astype(np.float32)
    step = rng.choice([-1, 0, 1], near.shape)          # one ulp below, on, or above the tie
    near = np.nextafter(near, np.where(step > 0, np.float32(np.inf), np.where(step < 0, np.float32(-np.inf), near)))
    blocks.append(np.concatenate([near, (127 * d)[:, None]], axis=1))   # amax pins d
    for b in blocks:
        b = b.astype(np.float32)
        xq = oracle.quantize_q8_1(b.reshape(1, -1)).reshape(len(b), 36)
        q_oracle = xq[:, 4:].view(np.int8).astype(np.int64)
        assert np.array_equal(_q8_fast_path(b), q_oracle)


def test_q4_0_unit_words_to_blocks():
    """The streaming kernel reads a 144-byte unit (eight 18-byte Q4_0 blocks) as 36
    aligned words w: block j (even) starts at word wa = 18 j / 4 with its scale in the
    low half of w[wa] and its nibbles two bytes into the next words, realigned by
    prmt(w[wa + i], w[wa + i + 1], 0x5432); block j + 1 has its scale in the high half
    of w[wa + 4] and its nibbles in w[wa + 5 .. wa + 8]."""
    rng = np.random.default_rng(41)
    for _ in range(200):
        unit = rng.integers(0, 256, 144, dtype=np.uint8)
        w = [int(v) for v in unit.view("<u4")]
        for j in range(0, 8, 2):
            wa = 18 * j // 4
            blk, nxt = unit[18 * j:18 * j + 18], unit[18 * j + 18:18 * j + 36]
            assert w[wa] & 0xFFFF == int(blk[:2].view("<u2")[0])
            assert w[wa + 4] >> 16 == int(nxt[:2].view("<u2")[0])
            for i in range(4):
                assert int(prmt(np.array([w[wa + i]]), np.array([w[wa + i + 1]]), 0x5432)[0]) == \
                    int(blk[2 + 4 * i:6 + 4 * i].view("<u4")[0])
                assert w[wa + 5 + i] == int(nxt[2 + 4 * i:6 + 4 * i].view("<u4")[0])


def test_q4_0_tensor_core_fragment_mapping():
    """mma.sync.m16n8k32.s8 fragments of the Q4_0 tensor-core kernel, lane (g, t) =
    (lane / 4, lane % 4): A registers {lo of row g, lo of row g + 8, hi of row g, hi of
    row g + 8} built from nibble word t of each row's block (k = 4t.. and 16 + 4t..),
    B registers Q8_1 words t and 4 + t of activation row g. Rebuilt into A (16 x 32)
    and B (32 x 8) by the PTX fragment layout, D = A B gives, in lane (g, t)'s d0..d3,
    16 (S - 8T) of weight rows g, g + 8 against activation rows 2t, 2t + 1."""
    qs, q8, S, T = _blocks(8, N=16, M=8, K=256)
    for b in range(qs.shape[1]):
        A = np.zeros((16, 32), np.int64)
        B = np.zeros((32, 8), np.int64)
        for lane in range(32):
            g, t = lane // 4, lane % 4
            lo = lambda r: ((qs[r, b, t] << 4) & 0xF0F0F0F0) ^ 0x80808080   # noqa: E731
            hi = lambda r: (qs[r, b, t] & 0xF0F0F0F0) ^ 0x80808080         # noqa: E731
            a = [lo(g), lo(g + 8), hi(g), hi(g + 8)]
            for j in range(4):
                A[g, 4 * t + j] = _s8(a[0])[j]
                A[g + 8, 4 * t + j] = _s8(a[1])[j]
                A[g, 16 + 4 * t + j] = _s8(a[2])[j]
                A[g + 8, 16 + 4 * t + j] = _s8(a[3])[j]
                B[4 * t + j, g] = _s8(q8[g, b, t])[j]
                B[16 + 4 * t + j, g] = _s8(q8[g, b, 4 + t])[j]
        D = A @ B
        want = 16 * (S[:, :, b] - 8 * T[:, None, b])    # [act][row]
        for lane in range(32):
            g, t = lane // 4, lane % 4
            d = [D[g, 2 * t], D[g, 2 * t + 1], D[g + 8, 2 * t], D[g + 8, 2 * t + 1]]
            assert d == [want[2 * t, g], want[2 * t + 1, g], want[2 * t, g + 8], want[2 * t + 1, g + 8]]

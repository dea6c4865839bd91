"""Shared-memory layout of the NVFP4/FP8 kernel's staged activations, checked on the
CPU: the B-fragment reads of every step are free of bank conflicts.

The activations of a pass are staged as M rows of fp16 with a row stride of
2 K + 16 bytes (16 mod 32) and 16-byte chunk c of a row stored at chunk
c ^ 2 ((c >> 3) & 3). Lane (g, t) = (lane / 4, lane % 4) of step s reads the
chunks s * (kStepK / 8) + kXChunks * t + i, i < kXChunks, of activation row
min(g + 8 mt, M - 1), 16 bytes at a time (kStepK = 256 k per step for NVFP4, 128
for FP8; kXChunks = kStepK / 32). A 16-byte shared-memory read is served eight
lanes at a time; it is conflict-free when those eight lanes touch eight different
16-byte bank groups (address / 16 mod 8), or the same address (a broadcast).
"""
import pytest


def row_stride(K):
    return 2 * K + 16


def chunk_slot(c):
    return c ^ (2 * ((c >> 3) & 3))


def conflicts(M, K, fp4):
    step_k = 256 if fp4 else 128
    x_chunks = step_k // 32
    rs = row_stride(K)
    bad = []
    for mt in (0, 1):
        for s in range(K // step_k):
            for i in range(x_chunks):
                addr = []
                for lane in range(32):
                    g, t = lane // 4, lane % 4
                    row = min(g + 8 * mt, M - 1)
                    c = s * (step_k // 8) + x_chunks * t + i
                    addr.append(row * rs + 16 * chunk_slot(c))
                for q in range(4):   # eight lanes at a time
                    a = addr[8 * q:8 * q + 8]
                    groups = {}
                    for x in a:
                        groups.setdefault((x // 16) % 8, set()).add(x)
                    if any(len(v) > 1 for v in groups.values()):
                        bad.append((mt, s, i, q))
    return bad


@pytest.mark.parametrize("fp4", [True, False])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 12, 16])
def test_activation_fragments_are_conflict_free(fp4, M):
    for K in (256, 1280, 5120):
        assert conflicts(M, K, fp4) == [], (M, K)


def test_without_the_swizzle_the_reads_conflict():
    """Control: with chunks stored in order the NVFP4 reads do collide (lanes of a
    quad read chunks 8 apart, which fall in one bank group)."""
    global chunk_slot
    saved = chunk_slot
    chunk_slot = lambda c: c   # noqa: E731
    try:
        assert conflicts(8, 5120, True)
    finally:
        chunk_slot = saved


def _constant(name):
    import os
    import re
    from conftest import ROOT
    src = open(os.path.join(ROOT, "gemm_qmv_quantize_gb300", "csrc", "q4_0_q8_1.cu")).read()
    return int(re.search(rf"constexpr int {name} = (\d+);", src).group(1))


@pytest.mark.parametrize("name,words", [("kActUnitStride", 21), ("kUnitBytes", 9)])
def test_q4_stream_records_and_units_are_conflict_free(name, words):
    """The Q4 streaming kernel: consecutive lanes read consecutive 144-byte weight
    units of a ring slot and consecutive 336-byte activation records of a row, 16 bytes
    at a time. Both strides are odd multiples of 16 bytes, so every 16-byte offset of
    eight consecutive units or records falls in eight different bank groups."""
    stride = _constant(name)
    assert stride == 16 * words and words % 2 == 1
    for j in range(words):
        for first in range(64):
            assert len({((first + l) * stride + 16 * j) // 16 % 8 for l in range(8)}) == 8

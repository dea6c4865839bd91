"""Pins of the oracle's fp32 -> Q8_1 quantizer.

- Hand-derived golden blocks (tests/golden/q8_1_blocks.json) covering ties,
  negative maxima, subnormal and large scales and the all-zero block.
- Invariants that hold for any input: |q| <= 127, q = +-127 at the element of
  largest magnitude, |x - d*q| <= d/2 (up to one fp32 ulp of x/d), s8 = fp16(d*sum q).
- An independent numpy restatement on random blocks, with round-half-away
  written as sign(v) * floor(|v| + 1/2) in fp64 (exact for any fp32 v).
"""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _cases():
    with open(os.path.join(GOLDEN, "q8_1_blocks.json")) as f:
        doc = json.load(f)
    by_name = {c["name"]: c for c in doc["cases"]}
    out = []
    for c in doc["cases"]:
        if "x" in c:
            x = np.array(c["x"], dtype=np.float32)
        else:
            x = np.array(by_name[c["x_from"]]["x"], dtype=np.float32) * np.float32(c["x_scale"])
        out.append((c["name"], x, c))
    return out


def _split(xq):
    d8 = xq[..., 0].astype(np.uint16) | (xq[..., 1].astype(np.uint16) << 8)
    s8 = xq[..., 2].astype(np.uint16) | (xq[..., 3].astype(np.uint16) << 8)
    q = xq[..., 4:36].view(np.int8)
    return d8, s8, q


@pytest.mark.parametrize("name,x,case", _cases(), ids=[c[0] for c in _cases()])
def test_golden_blocks(name, x, case):
    xq = oracle.quantize_q8_1(x[None, :]).reshape(1, 36)
    d8, s8, q = _split(xq)
    assert list(q[0]) == case["q"]
    assert int(d8[0]) == int(case["d8"], 16)
    assert int(s8[0]) == int(case["s8"], 16)


def test_layout_rows_and_blocks_independent():
    """A 2x64 input is four independent blocks laid out [m][b]."""
    cases = _cases()
    blocks = [cases[0][1], cases[1][1], cases[2][1], cases[4][1]]
    x = np.stack([np.concatenate(blocks[0:2]), np.concatenate(blocks[2:4])])
    xq = oracle.quantize_q8_1(x)
    for i, blk in enumerate(blocks):
        single = oracle.quantize_q8_1(blk[None, :])[0]
        m, b = divmod(i, 2)
        assert np.array_equal(xq[m, b * 36:(b + 1) * 36], single)


def _numpy_restatement(x):
    x = x.reshape(-1, 32).astype(np.float32)
    amax = np.max(np.abs(x), axis=1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (x / d[:, None]).astype(np.float32).astype(np.float64)
    q = np.sign(v) * np.floor(np.abs(v) + 0.5)
    q = np.where(d[:, None] == 0, 0, np.clip(q, -127, 127)).astype(np.int64)
    s = (d * q.sum(axis=1).astype(np.float32)).astype(np.float32)
    with np.errstate(over="ignore"):   # an s8 past 65504 is stored as inf, as in the oracle
        return d.astype(np.float16).view(np.uint16), s.astype(np.float16).view(np.uint16), q


@pytest.mark.parametrize("scale", [1.0, 1e-3, 37.0, 1e4])
def test_random_blocks_match_numpy_restatement(scale):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((3, 32 * 40)) * scale).astype(np.float32)
    # exact ties: make some elements land exactly on k + 1/2 after the division
    x[0, :32] = np.float32(127.0) * np.array([1.0] + [((k % 9) + 0.5) / 127.0 for k in range(31)],
                                              dtype=np.float32)
    xq = oracle.quantize_q8_1(x)
    d8, s8, q = _split(xq.reshape(3, 40, 36))
    rd8, rs8, rq = _numpy_restatement(x)
    assert np.array_equal(d8.reshape(-1), rd8)
    assert np.array_equal(s8.reshape(-1), rs8)
    assert np.array_equal(q.reshape(-1, 32).astype(np.int64), rq)


def test_invariants_on_random_input():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 32 * 64)).astype(np.float32)
    x[1] *= 1e-6
    x[2, ::7] = 0
    xq = oracle.quantize_q8_1(x).reshape(4, 64, 36)
    d8, s8, q = _split(xq)
    xb = x.reshape(4, 64, 32)
    amax = np.abs(xb).max(axis=2)
    d = (amax / np.float32(127)).astype(np.float32)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    # the element of largest magnitude quantizes to +-127
    arg = np.abs(xb).argmax(axis=2)
    qa = np.take_along_axis(q.astype(np.int32), arg[..., None], axis=2)[..., 0]
    xa = np.take_along_axis(xb, arg[..., None], axis=2)[..., 0]
    assert np.all(qa == np.sign(xa) * 127)
    # reconstruction error at most half a step (plus the fp32 rounding of x/d)
    err = np.abs(xb.astype(np.float64) - d[..., None].astype(np.float64) * q)
    assert np.all(err <= d[..., None] * (0.5 + 1e-6))
    # stored d8 is fp16(d), s8 is fp16(d * sum q)
    assert np.array_equal(d8, d.astype(np.float16).view(np.uint16))
    s = (d * q.astype(np.int32).sum(axis=2).astype(np.float32)).astype(np.float32)
    assert np.array_equal(s8, s.astype(np.float16).view(np.uint16))

"""Pins of the oracle's element decoders/encoders against library routines and closed forms.

fp16: IEEE 754 binary16, checked against numpy's float16 over every bit pattern and
over fp32 values chosen to hit ties, subnormals and the overflow boundary.
E4M3 / E2M1: the OCP MX v1.0 element definitions, checked against torch's
float8_e4m3fn decoder over all 256 codes and against the closed forms
(-1)^s 2^(e-bias) (1 + m/2^mbits) written independently here.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_fp16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the sign of zero survives
    assert math.copysign(1.0, oracle.fp16_to_double(0x8000)) == -1.0


def _fp16_edge_values():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, -65520.0, 70000.0, 1e30,
            2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 1.5 * 2.0 ** -24,
            2.5 * 2.0 ** -24, 5.96e-8, 6.1e-5, 0.1, 1 / 3]
    # exact ties between neighbouring binary16 values, both parities, normal and subnormal
    for base in (1.0, 2.0, 1024.0, 2.0 ** -14, 2.0 ** -20):
        ulp = np.spacing(np.float16(base)).astype(np.float64)
        for k in range(6):
            vals.append(base + (k + 0.5) * ulp)
            vals.append(-(base + (k + 0.5) * ulp))
    return vals


def test_fp16_encode_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        np.array(_fp16_edge_values(), dtype=np.float32),
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-5).astype(np.float32),
        (rng.standard_normal(5000) * 3e4).astype(np.float32),
        np.exp(rng.uniform(-20, 12, 20000)).astype(np.float32),
    ])
    with np.errstate(over="ignore"):   # values past 65504 become inf, as intended
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_fp16(v) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_fp16_encode_nan_and_inf():
    assert oracle.float_to_fp16(float("inf")) == 0x7C00
    assert oracle.float_to_fp16(float("-inf")) == 0xFC00
    assert (oracle.float_to_fp16(float("nan")) & 0x7C00) == 0x7C00
    assert (oracle.float_to_fp16(float("nan")) & 0x03FF) != 0


def _e4m3_closed_form(b: int) -> float:
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return math.nan
    mag = (m / 8.0) * 2.0 ** (1 - 7) if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def test_e4m3_decode_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = oracle.e4m3_to_double(b)
        cf = _e4m3_closed_form(b)
        if math.isnan(cf):
            assert math.isnan(got) and math.isnan(lib[b]), b
        else:
            assert got == cf == lib[b], (b, got, cf, lib[b])
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_double(0x38) == 1.0


def _e2m1_closed_form(c: int) -> float:
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2.0)
    return -mag if s else mag


def test_e2m1_table_closed_form():
    for c in range(16):
        assert oracle.e2m1_to_double(c) == _e2m1_closed_form(c), c
    mags = [oracle.e2m1_to_double(c) for c in range(8)]
    assert mags == sorted(mags) and len(set(mags)) == 8
    if hasattr(torch, "float4_e2m1fn_x2"):
        pass  # torch offers no element-wise decoder for the packed type; the closed form stands


def test_e2m1_round_trip():
    for c in range(16):
        back = oracle.e2m1_encode(oracle.e2m1_to_double(c))
        if c == 0x8:
            assert back in (0x0, 0x8)  # -0 and +0 are the same value
        else:
            assert back == c, (c, back)


@pytest.mark.parametrize("v,code", [(0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4),
                                    (3.5, 0x6), (5.0, 0x6), (7.0, 0x7), (-2.6, 0xD)])
def test_e2m1_encode_ties_to_even(v, code):
    assert oracle.e2m1_encode(v) == code


def test_e2m1_times_e4m3_is_exact_in_fp16():
    """The NVFP4 kernel folds the group scale into the fp16 weight (one fp16 multiply
    per pair): every E2M1 value times every non-NaN E4M3 scale has at most 6
    significant bits and a magnitude within [2^-10, 2688], so fp16 holds it exactly
    and the only rounding left is the fp32 accumulation."""
    vals = [oracle.e2m1_to_double(c) for c in range(16)]
    scales = [oracle.e4m3_to_double(b) for b in range(256) if b & 0x7F != 0x7F]
    nonzero = []
    for v in vals:
        for s in scales:
            p = v * s
            assert float(np.float16(p)) == p, (v, s)
            if p:
                nonzero.append(abs(p))
    assert min(nonzero) == 2.0 ** -10 and max(nonzero) == 6 * 448 == 2688

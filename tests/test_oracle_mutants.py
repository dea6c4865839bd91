"""Planted mistakes: each mutant is a copy of the oracle source with one
plausible error (a swapped nibble half, a dropped offset, a wrong scale group,
a transposed operand, ties to even instead of away from zero, an off-by-one
exponent bias, a signed maximum, a dropped global scale, a 5-bit mask). The oracle's pin tests must fail on every one of them.

The mistakes are planted in a temporary copy of the oracle on the CPU; the
oracle itself is never modified.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "qmv_oracle.c")
PIN_TESTS = ["tests/test_oracle_codecs.py", "tests/test_oracle_quantize.py",
             "tests/test_oracle_q4_0.py", "tests/test_oracle_nvfp4_fp8.py", "tests/test_oracle_q4_k.py"]

MUTANTS = {
    "q4_nibble_halves_swapped": ("(j < 16) ? (qs[j] & 0x0f) : (qs[j - 16] >> 4)",
                                 "(j < 16) ? (qs[j] >> 4) : (qs[j - 16] & 0x0f)"),
    "q4_offset_dropped": ("(double)(q4_0_nibble(wb + 2, j) - 8)",
                          "(double)(q4_0_nibble(wb + 2, j))"),
    "q4_scale_of_next_block": ("const uint8_t *wb = w + (n * nb + b) * 18;",
                               "const uint8_t *wb = w + (n * nb + (b + 1) % nb) * 18;"),
    "q8_ties_to_even": ("float r = roundf(xb[i] / d);", "float r = rintf(xb[i] / d);"),
    "q8_sum_from_d8": ("oracle_float_to_fp16(d * (float)sum)",
                       "oracle_float_to_fp16((float)oracle_fp16_to_double(d8) * (float)sum)"),
    "fp16_subnormal_unit": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "nvfp4_nibble_order": ("(k % 2 == 0) ? (uint8_t)(byte & 0x0f) : (uint8_t)(byte >> 4)",
                           "(k % 2 == 0) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0x0f)"),
    "nvfp4_scale_per_32": ("oracle_e4m3_to_double(scales[n * (K / 16) + k / 16])",
                           "oracle_e4m3_to_double(scales[n * (K / 16) + k / 32])"),
    "e4m3_bias": ("else v = ldexp((double)(8 + m), e - 10);", "else v = ldexp((double)(8 + m), e - 9);"),
    "e2m1_table": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 8.0}"),
    "q4k_min_sign": ("* (double)q4_k_nibble(blk + 16, i) - dmin * (double)mn;",
                     "* (double)q4_k_nibble(blk + 16, i) + dmin * (double)mn;"),
    "q4k_dmin_read_as_d": ("double dmin = oracle_fp16_to_double(read_u16le(blk + 2));",
                           "double dmin = oracle_fp16_to_double(read_u16le(blk));"),
    "q4k_scale_min_swapped": ("*sc = p[j] & 63;\n        *mn = p[j + 4] & 63;",
                              "*sc = p[j + 4] & 63;\n        *mn = p[j] & 63;"),
    "q4k_high_bits_from_wrong_byte": ("*sc = (p[j + 4] & 15) | ((p[j - 4] >> 6) << 4);",
                                      "*sc = (p[j + 4] & 15) | ((p[j] >> 6) << 4);"),
    "q4k_nibble_halves_swapped": ("(r < 32) ? (qs[32 * c + r] & 0x0f) : (qs[32 * c + r - 32] >> 4)",
                                  "(r < 32) ? (qs[32 * c + r] >> 4) : (qs[32 * c + r - 32] & 0x0f)"),
    "q4k_adjacent_nibble_pairs": ("(r < 32) ? (qs[32 * c + r] & 0x0f) : (qs[32 * c + r - 32] >> 4)",
                                  "(r % 2 == 0) ? (qs[32 * c + r / 2] & 0x0f) : (qs[32 * c + r / 2] >> 4)"),
    "q4k_sub_block_of_next": ("oracle_q4_k_scale_min(blk + 4, i / 32, &sc, &mn);",
                              "oracle_q4_k_scale_min(blk + 4, (i / 32 + 1) % 8, &sc, &mn);"),
    "q8_amax_signed": ("float a = fabsf(xb[i]);", "float a = xb[i];"),
    "q8_scale_over_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "q4_block_sum_t_drops_last": ("for (int j = 0; j < 32; ++j) t += q8[j];",
                                  "for (int j = 0; j < 31; ++j) t += q8[j];"),
    "nvfp4_global_scale_dropped": ("* (double)g;", "* 1.0;"),
    "fp8_row_scale_of_next_row": ("(double)rs[n]", "(double)rs[(n + 1) % N]"),
    "e4m3_subnormal_unit": ("if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp((double)m, -10);"),
    "q4k_min_high_bits_from_wrong_byte": ("*mn = (p[j + 4] >> 4) | ((p[j] >> 6) << 4);",
                                          "*mn = (p[j + 4] >> 4) | ((p[j - 4] >> 6) << 4);"),
    "q4k_scale_five_bits": ("*sc = p[j] & 63;", "*sc = p[j] & 31;"),
    "fp8_x_transposed": ("double xv = oracle_fp16_to_double(x[m * K + k]);\n                acc += wv * xv;\n                mag += fabs(wv * xv);\n            }\n            y[m * N + n] = acc;\n            bound[m * N + n] = mag;\n        }\n    }\n}\n",
                         "double xv = oracle_fp16_to_double(x[(k * M + m) % (M * K)]);\n                acc += wv * xv;\n                mag += fabs(wv * xv);\n            }\n            y[m * N + n] = acc;\n            bound[m * N + n] = mag;\n        }\n    }\n}\n"),
}


def _build_mutant(tmp, name, old, new):
    with open(SRC) as f:
        src = f.read()
    # the last occurrence: the FP8 routine is the file's last function
    idx = src.rfind(old)
    assert idx >= 0, f"mutation site of {name} not found"
    mutated = src[:idx] + new + src[idx + len(old):]
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"{name}.so")
    with open(c, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared", c, "-o", so, "-lm"],
                   check=True)
    return so


def _run_pins(so):
    env = dict(os.environ, QMV_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PIN_TESTS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-600:]


def test_pins_catch_every_planted_mistake(tmp_path):
    sos = {name: _build_mutant(str(tmp_path), name, old, new) for name, (old, new) in MUTANTS.items()}
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = dict(zip(sos, ex.map(_run_pins, sos.values())))
    survivors = {name: out for name, (rc, out) in results.items() if rc != 1}
    assert not survivors, survivors


def test_unmutated_copy_passes_pins(tmp_path):
    """Control: the same harness on an unmodified copy passes."""
    so = _build_mutant(str(tmp_path), "control", "#include <math.h>", "#include <math.h>")
    rc, out = _run_pins(so)
    assert rc == 0, out

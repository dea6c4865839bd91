"""Host-side checks of the C ABI that need no GPU.

- libqmv.so builds for sm_103a, loads, and exports every entry point that
  include/*.h declares (and the binding's signature table matches the header).
- Argument validation runs before any CUDA call: invalid shapes, NULL and
  misaligned pointers return their status codes and launch nothing. Only
  pointer values are passed (never dereferenced on the host).
"""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from gemm_qmv_quantize_gb300 import build
    build.build()
    import gemm_qmv_quantize_gb300 as q
    return q.lib()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as f:
            text = f.read()
        names |= set(re.findall(r"QMV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))
    return names


def test_header_declares_the_four_entry_points():
    names = _declared_symbols()
    for n in ("qmv_quantize_q8_1", "qmv_q4_0_q8_1", "qgemm_nvfp4_w4a16", "qgemm_fp8_w8a16"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_header_is_plain_c_and_links(lib, tmp_path):
    """A C99 program (no CUDA headers) that includes include/qmv.h, takes the address
    of every declared entry point, links against libqmv.so and runs calls that answer
    before any CUDA call."""
    import subprocess
    names = sorted(_declared_symbols())
    src = tmp_path / "abi_check.c"
    src.write_text("\n".join([
        "#include <stdio.h>",
        '#include "qmv.h"',
        "typedef void (*fn)(void);",
        "static const fn every[] = {" + ", ".join(f"(fn){n}" for n in names) + "};",
        "int main(void) {",
        "    int bad = 0;",
        "    if (sizeof every / sizeof every[0] != %d) bad |= 1;" % len(names),
        "    if (qmv_quantize_q8_1(0, 0, 1, 64, 0) != QMV_ERR_NULL) bad |= 2;",
        "    if (qmv_q4_0_q8_1((const void *)0x10000, (const void *)0x10000, (float *)0x10000, 9, 64, 4096, 0)"
        " != QMV_ERR_SHAPE) bad |= 4;",
        "    if (qmv_route_count() < 1 || !qmv_status_string(QMV_ERR_ALIGN)) bad |= 8;",
        '    printf("%d\\n", bad);',
        "    return bad;",
        "}", ""]))
    build_dir = os.path.dirname(lib._name)
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe), "-L", build_dir, "-lqmv", f"-Wl,-rpath,{build_dir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "0", (r.stdout, r.stderr)


def test_binding_table_matches_header():
    from gemm_qmv_quantize_gb300 import _binding
    assert set(_binding.SIGNATURES) == _declared_symbols()


def test_library_is_sm_103a(lib):
    from gemm_qmv_quantize_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


OK, NULL, SHAPE, ALIGN = 0, -1, -2, -3
P = 0x10000          # a 16-byte aligned fake pointer value (never dereferenced)


@pytest.mark.parametrize("args,status", [
    ((0, P, 1, 4096, None), NULL),
    ((P, 0, 1, 4096, None), NULL),
    ((P, P, 9, 4096, None), SHAPE),
    ((P, P, -1, 4096, None), SHAPE),
    ((P, P, 1, 4097, None), SHAPE),
    ((P + 2, P, 1, 4096, None), ALIGN),
    ((P, P + 1, 1, 4096, None), ALIGN),
    ((0, 0, 0, 4096, None), OK),     # M == 0: empty call
    ((0, 0, 1, 0, None), OK),        # K == 0: nothing to quantize
])
def test_quantize_validation(lib, args, status):
    assert lib.qmv_quantize_q8_1(*args) == status


@pytest.mark.parametrize("args,status", [
    ((0, P, P, 1, 64, 4096, None), NULL),
    ((P, 0, P, 1, 64, 4096, None), NULL),
    ((P, P, 0, 1, 64, 4096, None), NULL),
    ((P, P, P, 9, 64, 4096, None), SHAPE),
    ((P, P, P, 1, -5, 4096, None), SHAPE),
    ((P, P, P, 1, 64, 4100, None), SHAPE),
    ((P, P, P, 1, 1 << 32, 4096, None), SHAPE),
    ((P + 1, P, P, 1, 64, 4096, None), ALIGN),
    ((P, P + 2, P, 1, 64, 4096, None), ALIGN),
    ((P, P, P + 2, 1, 64, 4096, None), ALIGN),
    ((0, 0, 0, 1, 0, 4096, None), OK),    # N == 0
    ((0, 0, 0, 0, 64, 4096, None), OK),   # M == 0
])
def test_q4_0_validation(lib, args, status):
    assert lib.qmv_q4_0_q8_1(*args) == status


@pytest.mark.parametrize("fn", ["qmv_q4_k_q8_1", "qmv_q4_k_q8_1_fused", "qmv_debug_q4_k_block_dots"])
@pytest.mark.parametrize("args,status", [
    ((0, P, P, 1, 64, 4096, None), NULL),
    ((P, 0, P, 1, 64, 4096, None), NULL),
    ((P, P, P, 9, 64, 4096, None), SHAPE),
    ((P, P, P, 1, -5, 4096, None), SHAPE),
    ((P, P, P, 1, 64, 4128, None), SHAPE),     # K % 256
    ((P + 8, P, P, 1, 64, 4096, None), ALIGN),  # super-block rows need 16-byte alignment
    ((P, P, P + 2, 1, 64, 4096, None), ALIGN),
    ((0, 0, 0, 1, 0, 4096, None), OK),          # N == 0
    ((0, 0, 0, 0, 64, 4096, None), OK),         # M == 0
])
def test_q4_k_validation(lib, fn, args, status):
    assert getattr(lib, fn)(*args) == status


def test_q4_k_validation_null_output_and_x_alignment(lib):
    assert lib.qmv_q4_k_q8_1(P, P, 0, 1, 64, 4096, None) == NULL
    assert lib.qmv_debug_q4_k_block_dots(P, P, 0, 1, 64, 4096, None) == NULL
    assert lib.qmv_q4_k_q8_1(P, P + 2, P, 1, 64, 4096, None) == ALIGN        # Q8_1 needs 4 bytes
    assert lib.qmv_q4_k_q8_1_fused(P, P + 4, P, 1, 64, 4096, None) == ALIGN  # fp32 x needs 16 bytes
    arr = ctypes.c_void_p * 2
    n = (ctypes.c_int64 * 2)(64, 64)
    z = arr(P, P)
    assert lib.qmv_q4_k_q8_1_group(9, z, z, z, n, 1, 4096, None) == SHAPE
    assert lib.qmv_q4_k_q8_1_group(2, z, z, z, n, 1, 4128, None) == SHAPE
    assert lib.qmv_q4_k_q8_1_fused_group(2, arr(P, P + 8), z, z, n, 1, 4096, None) == ALIGN


@pytest.mark.parametrize("args,status", [
    ((0, P, 0.01, P, P, 1, 64, 512, None), NULL),
    ((P, 0, 0.01, P, P, 1, 64, 512, None), NULL),
    ((P, P, 0.01, 0, P, 1, 64, 512, None), NULL),
    ((P, P, 0.01, P, 0, 1, 64, 512, None), NULL),
    ((P, P, 0.01, P, P, 1, 64, 520, None), SHAPE),
    ((P, P, 0.01, P, P, 97, 64, 512, None), SHAPE),   # M > 96
    ((P, P, 0.01, P, P, -1, 64, 512, None), SHAPE),
    ((P, P, 0.01, P + 1, P, 1, 64, 512, None), ALIGN),
    ((P, P, 0.01, P, P + 2, 1, 64, 512, None), ALIGN),
    ((0, 0, 0.01, 0, 0, 1, 0, 512, None), OK),
])
def test_nvfp4_validation(lib, args, status):
    assert lib.qgemm_nvfp4_w4a16(*args) == status


@pytest.mark.parametrize("args,status", [
    ((0, P, P, P, 1, 64, 512, None), NULL),
    ((P, 0, P, P, 1, 64, 512, None), NULL),
    ((P, P, 0, P, 1, 64, 512, None), NULL),
    ((P, P, P, 0, 1, 64, 512, None), NULL),
    ((P, P, P, P, 1, 64, -1, None), SHAPE),
    ((P, P, P, P, 97, 64, 512, None), SHAPE),         # M > 96
    ((P, P + 2, P, P, 1, 64, 512, None), ALIGN),
    ((P, P, P + 1, P, 1, 64, 512, None), ALIGN),
    ((P, P, P, P + 1, 1, 64, 512, None), ALIGN),
])
def test_fp8_validation(lib, args, status):
    assert lib.qgemm_fp8_w8a16(*args) == status


@pytest.mark.parametrize("fn", ["qmv_q4_0_q8_1_fused_group", "qmv_q4_0_q8_1_group"])
def test_group_validation(lib, fn):
    import ctypes
    arr = ctypes.c_void_p * 9
    n = (ctypes.c_int64 * 9)(*([64] * 9))
    z = arr(*([P] * 9))
    f = getattr(lib, f"{fn}")
    assert f(9, z, z, z, n, 1, 4096, None) == SHAPE        # count > 8
    assert f(0, z, z, z, n, 1, 4096, None) == SHAPE
    assert f(2, z, z, z, n, 1, 4000, None) == SHAPE        # K % 256
    assert f(2, z, z, z, n, 9, 4096, None) == SHAPE        # M > 8
    assert f(2, None, z, z, n, 1, 4096, None) == NULL
    assert f(2, arr(P, P + 8), z, z, n, 1, 4096, None) == ALIGN     # w not 16-aligned
    assert f(2, z, z, arr(P, P + 2), n, 1, 4096, None) == ALIGN     # y not 4-aligned
    assert f(2, z, z, z, n, 0, 4096, None) == OK           # M == 0
    x_off = 4 if fn == "qmv_q4_0_q8_1_group" else 16       # Q8_1 needs 4 bytes, fp32 fused 16
    assert f(2, z, arr(P, P + 2), z, n, 1, 4096, None) == ALIGN
    assert f(2, z, arr(P, P + x_off // 2), z, n, 1, 4096, None) == ALIGN


def test_wq_group_validation(lib):
    import ctypes
    arr = ctypes.c_void_p * 9
    n = (ctypes.c_int64 * 9)(*([64] * 9))
    z = arr(*([P] * 9))
    g = (ctypes.c_float * 9)(*([0.01] * 9))
    nv, f8 = lib.qgemm_nvfp4_w4a16_group, lib.qgemm_fp8_w8a16_group
    assert nv(9, z, z, g, P, z, n, 1, 512, None) == SHAPE           # count > 8
    assert nv(2, z, z, g, P, z, n, 1, 528, None) == SHAPE           # K % 256 (the tensor-core kernel only)
    assert nv(2, z, z, None, P, z, n, 1, 512, None) == NULL         # no global scales
    assert nv(2, arr(P, P + 8), z, g, P, z, n, 1, 512, None) == ALIGN   # codes not 16-aligned
    assert nv(2, z, z, g, P + 8, z, n, 1, 512, None) == ALIGN       # x not 16-aligned
    assert nv(2, z, z, g, P, z, n, 0, 512, None) == OK              # M == 0
    assert f8(2, z, z, P, z, n, 1, 200, None) == SHAPE              # K % 128
    assert f8(2, z, arr(P, P + 2), P, z, n, 1, 384, None) == ALIGN  # row scale not 4-aligned
    assert f8(9, z, z, P, z, n, 1, 384, None) == SHAPE
    assert nv(2, z, z, g, P, z, n, 97, 512, None) == SHAPE          # M > 96
    assert f8(2, z, z, P, z, n, 97, 384, None) == SHAPE


def test_debug_dots_validation(lib):
    assert lib.qmv_debug_q4_0_block_dots(P, P, 0, 1, 64, 4096, None) == NULL
    assert lib.qmv_debug_q4_0_block_dots(P, P, P, 9, 64, 4096, None) == SHAPE


def test_status_strings_and_routes(lib):
    for s in (OK, NULL, SHAPE, ALIGN, -4, -5, 123):
        assert lib.qmv_status_string(s)
    n = lib.qmv_route_count()
    names = [lib.qmv_route_name(i).decode() for i in range(n)]
    assert len(set(names)) == n and "q4_0_stream_dp4a" in names
    lib.qmv_route_reset()
    assert all(lib.qmv_route_launches(i) == 0 for i in range(n))
    assert lib.qmv_route_launches(n) == -1


def test_error_flags_null(lib):
    assert lib.qmv_error_flags(None, 0) == NULL


def test_wait_bound_validation(lib):
    assert lib.qmv_debug_wait_bound(None, None) == NULL
    assert lib.qmv_debug_wait_bound(P + 4, None) == ALIGN


def test_cta_abort_validation(lib):
    assert lib.qmv_debug_cta_abort(None, 3, None) == NULL
    assert lib.qmv_debug_cta_abort(P + 4, 3, None) == ALIGN
    assert lib.qmv_debug_cta_abort(P, -1, None) == SHAPE
    assert lib.qmv_debug_cta_abort(P, 8, None) == SHAPE


def test_binding_raises_loudly_when_library_missing(monkeypatch, tmp_path):
    from gemm_qmv_quantize_gb300 import _binding
    monkeypatch.setattr(_binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(_binding.QmvLibraryMissing):
        _binding.lib()

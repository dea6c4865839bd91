"""CPU oracle for the quantized skinny matmul path (ctypes wrapper over qmv_oracle.c).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. It
shares no code with the CUDA path and never imports it.

All functions take and return numpy arrays on the host. Floating-point results
are fp64 (``y``) together with ``bound`` = sum_k |w * x| per output, the scale of
the parity tolerance |y_gpu - y| <= 1e-3 * bound + 1e-6.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

_lock = threading.Lock()
_handle = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def _lib():
    """The oracle library; ``QMV_ORACLE_LIB`` names another build of
    qmv_oracle.c (the planted-mistake builds of the pin tests)."""
    global _handle
    with _lock:
        if _handle is None:
            _handle = _load(os.environ.get("QMV_ORACLE_LIB") or _build.build())
    return _handle


def _load(path):
    lib = ctypes.CDLL(path)
    lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_double.restype = ctypes.c_double
    lib.oracle_float_to_fp16.argtypes = [ctypes.c_float]
    lib.oracle_float_to_fp16.restype = ctypes.c_uint16
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_to_double.restype = ctypes.c_double
    lib.oracle_e2m1_encode.argtypes = [ctypes.c_double]
    lib.oracle_e2m1_encode.restype = ctypes.c_uint8
    lib.oracle_quantize_q8_1.argtypes = [_f32p, _u8p, _i64, _i64]
    lib.oracle_quantize_q8_1.restype = None
    lib.oracle_q4_0_block_dots.argtypes = [_u8p, _u8p, _i64, _i64, _i64, _i32p, _i32p]
    lib.oracle_q4_0_block_dots.restype = None
    lib.oracle_q4_0_q8_1.argtypes = [_u8p, _u8p, _i64, _i64, _i64, _f64p, _f64p]
    lib.oracle_q4_0_q8_1.restype = None
    lib.oracle_nvfp4_w4a16.argtypes = [_u8p, _u8p, ctypes.c_float, _u16p, _i64, _i64,
                                       _i64, _f64p, _f64p]
    lib.oracle_nvfp4_w4a16.restype = None
    lib.oracle_fp8_w8a16.argtypes = [_u8p, _f32p, _u16p, _i64, _i64, _i64, _f64p, _f64p]
    lib.oracle_fp8_w8a16.restype = None
    lib.oracle_q4_k_scale_min.argtypes = [_u8p, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(ctypes.c_int)]
    lib.oracle_q4_k_scale_min.restype = None
    lib.oracle_q4_k_weight.argtypes = [_u8p, ctypes.c_int]
    lib.oracle_q4_k_weight.restype = ctypes.c_double
    lib.oracle_q4_k_block_dots.argtypes = [_u8p, _u8p, _i64, _i64, _i64, _i32p]
    lib.oracle_q4_k_block_dots.restype = None
    lib.oracle_q4_k_q8_1.argtypes = [_u8p, _u8p, _i64, _i64, _i64, _f64p, _f64p]
    lib.oracle_q4_k_q8_1.restype = None
    return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


# ---------------------------------------------------------------- element codecs

def fp16_to_double(bits: int) -> float:
    return _lib().oracle_fp16_to_double(int(bits))


def float_to_fp16(v: float) -> int:
    """fp32 value -> binary16 bit pattern (round to nearest even)."""
    return int(_lib().oracle_float_to_fp16(float(np.float32(v))))


def e4m3_to_double(b: int) -> float:
    return _lib().oracle_e4m3_to_double(int(b))


def e2m1_to_double(c: int) -> float:
    return _lib().oracle_e2m1_to_double(int(c))


def e2m1_encode(v: float) -> int:
    return int(_lib().oracle_e2m1_encode(float(v)))


# ---------------------------------------------------------------- the path

def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """fp32 [M][K] -> Q8_1 bytes [M][K/32*36]."""
    x = _as(x, np.float32)
    M, K = x.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    xq = np.zeros((M, K // 32 * 36), dtype=np.uint8)
    _lib().oracle_quantize_q8_1(_ptr(x, ctypes.c_float), _ptr(xq, ctypes.c_uint8), M, K)
    return xq


def q4_0_block_dots(w: np.ndarray, xq: np.ndarray, K: int):
    """Integer block sums: S [M][N][K/32] = sum q4u*q8, T [M][K/32] = sum q8."""
    w = _as(w, np.uint8)
    xq = _as(xq, np.uint8)
    N, M, nb = w.shape[0], xq.shape[0], K // 32
    assert w.shape[1] == nb * 18 and xq.shape[1] == nb * 36
    S = np.zeros((M, N, nb), dtype=np.int32)
    T = np.zeros((M, nb), dtype=np.int32)
    _lib().oracle_q4_0_block_dots(_ptr(w, ctypes.c_uint8), _ptr(xq, ctypes.c_uint8), M, N, K,
                                  _ptr(S, ctypes.c_int32), _ptr(T, ctypes.c_int32))
    return S, T


def q4_0_q8_1(w: np.ndarray, xq: np.ndarray, K: int):
    """y [M][N] (fp64) and bound [M][N] for Q4_0 weights against Q8_1 activations."""
    w = _as(w, np.uint8)
    xq = _as(xq, np.uint8)
    N, M, nb = w.shape[0], xq.shape[0], K // 32
    assert w.shape[1] == nb * 18 and xq.shape[1] == nb * 36
    y = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    _lib().oracle_q4_0_q8_1(_ptr(w, ctypes.c_uint8), _ptr(xq, ctypes.c_uint8), M, N, K,
                            _ptr(y, ctypes.c_double), _ptr(bound, ctypes.c_double))
    return y, bound


def nvfp4_w4a16(codes: np.ndarray, scales: np.ndarray, g: float, x_f16: np.ndarray):
    """y [M][N] (fp64) and bound for NVFP4 weights against fp16 activations.

    ``x_f16`` may be a numpy float16 array or its uint16 bit patterns.
    """
    codes = _as(codes, np.uint8)
    scales = _as(scales, np.uint8)
    x = np.ascontiguousarray(np.asarray(x_f16).view(np.uint16))
    M, K = x.shape
    N = codes.shape[0]
    assert codes.shape[1] == K // 2 and scales.shape == (N, K // 16)
    y = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    _lib().oracle_nvfp4_w4a16(_ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                              float(g), _ptr(x, ctypes.c_uint16), M, N, K,
                              _ptr(y, ctypes.c_double), _ptr(bound, ctypes.c_double))
    return y, bound


def fp8_w8a16(w: np.ndarray, row_scale: np.ndarray, x_f16: np.ndarray):
    """y [M][N] (fp64) and bound for FP8 E4M3 weights with per-row fp32 scale."""
    w = _as(w, np.uint8)
    rs = _as(row_scale, np.float32)
    x = np.ascontiguousarray(np.asarray(x_f16).view(np.uint16))
    M, K = x.shape
    N = w.shape[0]
    assert w.shape[1] == K and rs.shape == (N,)
    y = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    _lib().oracle_fp8_w8a16(_ptr(w, ctypes.c_uint8), _ptr(rs, ctypes.c_float),
                            _ptr(x, ctypes.c_uint16), M, N, K,
                            _ptr(y, ctypes.c_double), _ptr(bound, ctypes.c_double))
    return y, bound


# ---------------------------------------------------------------- Q4_K

def q4_k_scale_min(packed12: np.ndarray, j: int):
    """(sc, mn) of sub-block j from the 12 packed scale bytes of a Q4_K super-block."""
    p = _as(packed12, np.uint8)
    assert p.shape == (12,)
    sc, mn = ctypes.c_int(), ctypes.c_int()
    _lib().oracle_q4_k_scale_min(_ptr(p, ctypes.c_uint8), int(j), ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def q4_k_dequantize(w: np.ndarray, K: int) -> np.ndarray:
    """Q4_K [N][K/256*144] bytes -> fp64 weights [N][K] (element by element)."""
    w = _as(w, np.uint8)
    N, nsb = w.shape[0], K // 256
    assert w.shape[1] == nsb * 144
    lib = _lib()
    out = np.zeros((N, K), dtype=np.float64)
    for n in range(N):
        for s in range(nsb):
            blk = np.ascontiguousarray(w[n, s * 144:(s + 1) * 144])
            bp = _ptr(blk, ctypes.c_uint8)
            for i in range(256):
                out[n, s * 256 + i] = lib.oracle_q4_k_weight(bp, i)
    return out


def q4_k_block_dots(w: np.ndarray, xq: np.ndarray, K: int) -> np.ndarray:
    """Integer sub-block sums S [M][N][K/32] = sum q4u*q8 (q4u the unsigned nibble)."""
    w = _as(w, np.uint8)
    xq = _as(xq, np.uint8)
    N, M, nb = w.shape[0], xq.shape[0], K // 32
    assert K % 256 == 0 and w.shape[1] == K // 256 * 144 and xq.shape[1] == nb * 36
    S = np.zeros((M, N, nb), dtype=np.int32)
    _lib().oracle_q4_k_block_dots(_ptr(w, ctypes.c_uint8), _ptr(xq, ctypes.c_uint8), M, N, K,
                                  _ptr(S, ctypes.c_int32))
    return S


def q4_k_q8_1(w: np.ndarray, xq: np.ndarray, K: int):
    """y [M][N] (fp64) and bound [M][N] for Q4_K weights against Q8_1 activations."""
    w = _as(w, np.uint8)
    xq = _as(xq, np.uint8)
    N, M, nb = w.shape[0], xq.shape[0], K // 32
    assert K % 256 == 0 and w.shape[1] == K // 256 * 144 and xq.shape[1] == nb * 36
    y = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    _lib().oracle_q4_k_q8_1(_ptr(w, ctypes.c_uint8), _ptr(xq, ctypes.c_uint8), M, N, K,
                            _ptr(y, ctypes.c_double), _ptr(bound, ctypes.c_double))
    return y, bound

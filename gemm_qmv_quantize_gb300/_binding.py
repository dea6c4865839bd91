"""ctypes binding of libqmv.so (include/qmv.h): argument marshalling only.

Every function takes torch tensors on the current CUDA device, checks dtype,
shape and contiguity, passes raw pointers and sizes to the C entry point of the
same name, and raises ``QmvError`` on a non-zero status. All arithmetic runs in
the library's CUDA kernels; there is no CPU path. If the library is missing the
first call raises ``QmvLibraryMissing`` (build it with ``__graft_entry__.build()``
or ``python -m gemm_qmv_quantize_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libqmv.so")
_lock = threading.Lock()
_lib = None

QMV_OK = 0
STATUS_NAMES = {0: "QMV_OK", -1: "QMV_ERR_NULL", -2: "QMV_ERR_SHAPE", -3: "QMV_ERR_ALIGN",
                -4: "QMV_ERR_CUDA", -5: "QMV_ERR_TIMEOUT"}

# name -> (restype, argtypes), mirroring include/qmv.h
_vp, _i32, _i64, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
SIGNATURES = {
    "qmv_status_string": (ctypes.c_char_p, [_i32]),
    "qmv_quantize_q8_1": (_i32, [_vp, _vp, _i32, _i64, _vp]),
    "qmv_q4_0_q8_1": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qmv_q4_0_q8_1_fused": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qmv_q4_0_q8_1_fused_group": (_i32, [_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         ctypes.POINTER(_i64), _i32, _i64, _vp]),
    "qmv_q4_0_q8_1_group": (_i32, [_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                   ctypes.POINTER(_i64), _i32, _i64, _vp]),
    "qgemm_nvfp4_w4a16": (_i32, [_vp, _vp, _f32, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qgemm_fp8_w8a16": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qgemm_nvfp4_w4a16_group": (_i32, [_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_f32), _vp,
                                       ctypes.POINTER(_vp), ctypes.POINTER(_i64), _i32, _i64, _vp]),
    "qgemm_fp8_w8a16_group": (_i32, [_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, ctypes.POINTER(_vp),
                                     ctypes.POINTER(_i64), _i32, _i64, _vp]),
    "qmv_debug_q4_0_block_dots": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qmv_q4_k_q8_1": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qmv_q4_k_q8_1_fused": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qmv_q4_k_q8_1_group": (_i32, [_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                   ctypes.POINTER(_i64), _i32, _i64, _vp]),
    "qmv_q4_k_q8_1_fused_group": (_i32, [_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         ctypes.POINTER(_i64), _i32, _i64, _vp]),
    "qmv_debug_q4_k_block_dots": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _vp]),
    "qmv_set_launch_overlap": (None, [_i32]),
    "qmv_get_launch_overlap": (_i32, []),
    "qmv_route_count": (_i32, []),
    "qmv_route_name": (ctypes.c_char_p, [_i32]),
    "qmv_route_launches": (_i64, [_i32]),
    "qmv_route_reset": (None, []),
    "qmv_error_flags": (_i32, [ctypes.POINTER(ctypes.c_uint32), _i32]),
    "qmv_debug_wait_bound": (_i32, [_vp, _vp]),
    "qmv_debug_cta_abort": (_i32, [_vp, _i32, _vp]),
    "qmv_debug_plan_wq": (_i32, [_i32, _i32, _i64, _i32, ctypes.POINTER(_i64), _i32, _i32, _i32, _i32,
                                 ctypes.POINTER(_i32), _vp]),
    "qmv_debug_plan_q4": (_i32, [_i32, _i32, _i64, _i64, _i32, _i32, _i32, _i32, _i32, _vp]),
}


class QmvLibraryMissing(RuntimeError):
    pass


class QmvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({lib().qmv_status_string(status).decode()})")


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libqmv.so (loaded once; raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise QmvLibraryMissing(
                    f"{_LIB_PATH} not found: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            handle = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _check(fn: str, status: int):
    if status != QMV_OK:
        raise QmvError(fn, status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def qmv_quantize_q8_1(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 [M, K] -> Q8_1 uint8 [M, K/32*36]."""
    _need(x, "x", torch.float32)
    M, K = x.shape
    if out is None:
        out = torch.empty((M, K // 32 * 36), dtype=torch.uint8, device=x.device)
    _need(out, "out", torch.uint8, (M, K // 32 * 36))
    _check("qmv_quantize_q8_1", lib().qmv_quantize_q8_1(x.data_ptr(), out.data_ptr(), M, K, _stream(stream)))
    return out


def qmv_q4_0_q8_1(w: torch.Tensor, xq: torch.Tensor, K: int, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Q4_0 uint8 [N, K/32*18] x Q8_1 uint8 [M, K/32*36] -> fp32 [M, N]."""
    N, M = w.shape[0], xq.shape[0]
    _need(w, "w", torch.uint8, (N, K // 32 * 18))
    _need(xq, "xq", torch.uint8, (M, K // 32 * 36))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=w.device)
    _need(out, "out", torch.float32, (M, N))
    _check("qmv_q4_0_q8_1", lib().qmv_q4_0_q8_1(w.data_ptr(), xq.data_ptr(), out.data_ptr(), M, N, K,
                                                _stream(stream)))
    return out


def qmv_q4_0_q8_1_fused(w: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Q4_0 uint8 [N, K/32*18] x fp32 [M, K] (quantized to Q8_1 in-kernel) -> fp32 [M, N]."""
    _need(x, "x", torch.float32)
    M, K = x.shape
    N = w.shape[0]
    _need(w, "w", torch.uint8, (N, K // 32 * 18))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, "out", torch.float32, (M, N))
    _check("qmv_q4_0_q8_1_fused", lib().qmv_q4_0_q8_1_fused(w.data_ptr(), x.data_ptr(), out.data_ptr(), M, N, K,
                                                            _stream(stream)))
    return out


def qmv_q4_0_q8_1_fused_group(ws, xs, outs=None, stream=None):
    """Several independent fused calls (same M, K) in one launch; returns the outputs."""
    count = len(ws)
    if count != len(xs) or not 1 <= count <= 8:
        raise ValueError("need 1..8 matrices and as many activations")
    M, K = xs[0].shape
    Ns = [w.shape[0] for w in ws]
    for i, (w, x) in enumerate(zip(ws, xs)):
        _need(x, f"x[{i}]", torch.float32, (M, K))
        _need(w, f"w[{i}]", torch.uint8, (Ns[i], K // 32 * 18))
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.float32, device=xs[0].device) for n in Ns]
    for i, o in enumerate(outs):
        _need(o, f"out[{i}]", torch.float32, (M, Ns[i]))
    arr = ctypes.c_void_p * count
    wp, xp, yp = arr(*[w.data_ptr() for w in ws]), arr(*[x.data_ptr() for x in xs]), arr(*[o.data_ptr() for o in outs])
    npa = (ctypes.c_int64 * count)(*Ns)
    _check("qmv_q4_0_q8_1_fused_group",
           lib().qmv_q4_0_q8_1_fused_group(count, wp, xp, yp, npa, M, K, _stream(stream)))
    return outs


def qmv_q4_0_q8_1_group(ws, xqs, K: int, outs=None, stream=None):
    """Several independent calls on Q8_1 activations (same M, K) in one launch."""
    count = len(ws)
    if count != len(xqs) or not 1 <= count <= 8:
        raise ValueError("need 1..8 matrices and as many activations")
    M = xqs[0].shape[0]
    Ns = [w.shape[0] for w in ws]
    for i, (w, xq) in enumerate(zip(ws, xqs)):
        _need(xq, f"xq[{i}]", torch.uint8, (M, K // 32 * 36))
        _need(w, f"w[{i}]", torch.uint8, (Ns[i], K // 32 * 18))
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.float32, device=xqs[0].device) for n in Ns]
    for i, o in enumerate(outs):
        _need(o, f"out[{i}]", torch.float32, (M, Ns[i]))
    arr = ctypes.c_void_p * count
    wp, xp, yp = arr(*[w.data_ptr() for w in ws]), arr(*[x.data_ptr() for x in xqs]), arr(*[o.data_ptr() for o in outs])
    npa = (ctypes.c_int64 * count)(*Ns)
    _check("qmv_q4_0_q8_1_group", lib().qmv_q4_0_q8_1_group(count, wp, xp, yp, npa, M, K, _stream(stream)))
    return outs


def qmv_debug_q4_0_block_dots(w: torch.Tensor, xq: torch.Tensor, K: int, out: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """int32 [M, N, K/32]: S - 8T per block, from the product kernel's device code."""
    N, M = w.shape[0], xq.shape[0]
    _need(w, "w", torch.uint8, (N, K // 32 * 18))
    _need(xq, "xq", torch.uint8, (M, K // 32 * 36))
    if out is None:
        out = torch.empty((M, N, K // 32), dtype=torch.int32, device=w.device)
    _need(out, "out", torch.int32, (M, N, K // 32))
    _check("qmv_debug_q4_0_block_dots",
           lib().qmv_debug_q4_0_block_dots(w.data_ptr(), xq.data_ptr(), out.data_ptr(), M, N, K, _stream(stream)))
    return out


# ---------------------------------------------------------------- Q4_K (144-byte super-blocks: same row bytes as Q4_0)

def qmv_q4_k_q8_1(w: torch.Tensor, xq: torch.Tensor, K: int, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Q4_K uint8 [N, K/256*144] x Q8_1 uint8 [M, K/32*36] -> fp32 [M, N]."""
    N, M = w.shape[0], xq.shape[0]
    _need(w, "w", torch.uint8, (N, K // 256 * 144))
    _need(xq, "xq", torch.uint8, (M, K // 32 * 36))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=w.device)
    _need(out, "out", torch.float32, (M, N))
    _check("qmv_q4_k_q8_1", lib().qmv_q4_k_q8_1(w.data_ptr(), xq.data_ptr(), out.data_ptr(), M, N, K,
                                                _stream(stream)))
    return out


def qmv_q4_k_q8_1_fused(w: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Q4_K uint8 [N, K/256*144] x fp32 [M, K] (quantized to Q8_1 in-kernel) -> fp32 [M, N]."""
    _need(x, "x", torch.float32)
    M, K = x.shape
    N = w.shape[0]
    _need(w, "w", torch.uint8, (N, K // 256 * 144))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, "out", torch.float32, (M, N))
    _check("qmv_q4_k_q8_1_fused", lib().qmv_q4_k_q8_1_fused(w.data_ptr(), x.data_ptr(), out.data_ptr(), M, N, K,
                                                            _stream(stream)))
    return out


def _q4_k_group(fn: str, ws, xs, K: int, fused: bool, outs, stream):
    count = len(ws)
    if count != len(xs) or not 1 <= count <= 8:
        raise ValueError("need 1..8 matrices and as many activations")
    M = xs[0].shape[0]
    Ns = [w.shape[0] for w in ws]
    for i, (w, x) in enumerate(zip(ws, xs)):
        if fused:
            _need(x, f"x[{i}]", torch.float32, (M, K))
        else:
            _need(x, f"xq[{i}]", torch.uint8, (M, K // 32 * 36))
        _need(w, f"w[{i}]", torch.uint8, (Ns[i], K // 256 * 144))
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.float32, device=xs[0].device) for n in Ns]
    for i, o in enumerate(outs):
        _need(o, f"out[{i}]", torch.float32, (M, Ns[i]))
    arr = ctypes.c_void_p * count
    wp, xp, yp = arr(*[w.data_ptr() for w in ws]), arr(*[x.data_ptr() for x in xs]), arr(*[o.data_ptr() for o in outs])
    npa = (ctypes.c_int64 * count)(*Ns)
    _check(fn, getattr(lib(), fn)(count, wp, xp, yp, npa, M, K, _stream(stream)))
    return outs


def qmv_q4_k_q8_1_group(ws, xqs, K: int, outs=None, stream=None):
    """Several independent Q4_K calls on Q8_1 activations (same M, K) in one launch."""
    return _q4_k_group("qmv_q4_k_q8_1_group", ws, xqs, K, False, outs, stream)


def qmv_q4_k_q8_1_fused_group(ws, xs, outs=None, stream=None):
    """Several independent fused Q4_K calls (same M, K) in one launch."""
    return _q4_k_group("qmv_q4_k_q8_1_fused_group", ws, xs, xs[0].shape[1], True, outs, stream)


def qmv_debug_wait_bound(out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int64 [2] on the current device: [1 if the bounded wait completed else 0,
    nanoseconds waited]; the wait is on an mbarrier nothing completes, so it gives up
    and sets the timeout bit of error_flags()."""
    if out is None:
        out = torch.full((2,), -1, dtype=torch.int64, device="cuda")
    _need(out, "out", torch.int64, (2,))
    _check("qmv_debug_wait_bound", lib().qmv_debug_wait_bound(out.data_ptr(), _stream(stream)))
    return out


def qmv_debug_cta_abort(stuck_warp: int = 3, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int64 [8][4] on the current device, per warp of the self-check CTA: [1 if its
    bounded wait gave up, 1 if it passed the round's barrier and saw the CTA's abort
    word, copies in flight when it left the round, nanoseconds from its first wait to
    the barrier]. Warp `stuck_warp` waits on copies that were never issued."""
    if out is None:
        out = torch.full((8, 4), -1, dtype=torch.int64, device="cuda")
    _need(out, "out", torch.int64, (8, 4))
    _check("qmv_debug_cta_abort", lib().qmv_debug_cta_abort(out.data_ptr(), int(stuck_warp), _stream(stream)))
    return out


PLAN_FIELDS = ("route", "warps", "slots", "grid", "smem_bytes", "act_regs", "pair", "chunk_units")
GB300_DEVICE = dict(sm_count=152, smem_optin=232448, smem_per_sm=233472)


def qmv_debug_plan_q4(M: int, N: int, K: int, q4k: bool = False, n_inputs: int = 1, w_align16: bool = True,
                      sm_count: int = GB300_DEVICE["sm_count"], smem_optin: int = GB300_DEVICE["smem_optin"],
                      smem_per_sm: int = GB300_DEVICE["smem_per_sm"]) -> dict:
    """The Q4_0 / Q4_K launch plan for one call on the given device (GB300 by
    default), as a dict of PLAN_FIELDS with the route as its name. No GPU needed for
    the streaming-kernel plans."""
    out = (ctypes.c_int64 * 8)()
    _check("qmv_debug_plan_q4", lib().qmv_debug_plan_q4(int(bool(q4k)), M, N, K, n_inputs, int(bool(w_align16)),
                                                        sm_count, smem_optin, smem_per_sm, out))
    plan = dict(zip(PLAN_FIELDS, (int(v) for v in out)))
    plan["route"] = lib().qmv_route_name(plan["route"]).decode()
    return plan


WQ_PLAN_FIELDS = ("route", "chunks", "chunk_rows", "warps", "slots", "staged", "passes", "tiles_per_round",
                  "ctas_per_sm", "grid", "smem_bytes", "a_bufs", "b_bufs", "k_splits")


def qmv_debug_plan_wq(M: int, K: int, N, fp4: bool = True, aligned16: bool = True, ctas_by_regs=None,
                      sm_count: int = GB300_DEVICE["sm_count"], smem_optin: int = GB300_DEVICE["smem_optin"],
                      smem_per_sm: int = GB300_DEVICE["smem_per_sm"]) -> dict:
    """The NVFP4 (fp4) / FP8 launch plan for one call (N an int) or one grouped launch
    (N a list of row counts) on the given device (GB300 by default), with CTAs per SM
    from the occupancy model of include/qmv.h; a dict of WQ_PLAN_FIELDS with the route
    as its name. No GPU needed."""
    Ns = [int(N)] if isinstance(N, int) else [int(n) for n in N]
    n_arr = (ctypes.c_int64 * len(Ns))(*Ns)
    regs = None if ctas_by_regs is None else (ctypes.c_int * 3)(*[int(v) for v in ctas_by_regs])
    out = (ctypes.c_int64 * len(WQ_PLAN_FIELDS))()
    _check("qmv_debug_plan_wq", lib().qmv_debug_plan_wq(int(bool(fp4)), M, K, len(Ns), n_arr, int(bool(aligned16)),
                                                        sm_count, smem_optin, smem_per_sm, regs, out))
    plan = dict(zip(WQ_PLAN_FIELDS, (int(v) for v in out)))
    plan["route"] = lib().qmv_route_name(plan["route"]).decode()
    return plan


def qmv_debug_q4_k_block_dots(w: torch.Tensor, xq: torch.Tensor, K: int, out: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """int32 [M, N, K/32]: raw S = sum q * q8 per sub-block, from the product kernel's device code."""
    N, M = w.shape[0], xq.shape[0]
    _need(w, "w", torch.uint8, (N, K // 256 * 144))
    _need(xq, "xq", torch.uint8, (M, K // 32 * 36))
    if out is None:
        out = torch.empty((M, N, K // 32), dtype=torch.int32, device=w.device)
    _need(out, "out", torch.int32, (M, N, K // 32))
    _check("qmv_debug_q4_k_block_dots",
           lib().qmv_debug_q4_k_block_dots(w.data_ptr(), xq.data_ptr(), out.data_ptr(), M, N, K, _stream(stream)))
    return out


def qgemm_nvfp4_w4a16(codes: torch.Tensor, scales: torch.Tensor, global_scale: float, x: torch.Tensor,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """NVFP4 codes uint8 [N, K/2], E4M3 scales uint8 [N, K/16], x fp16 [M, K] -> fp32 [M, N]."""
    _need(x, "x", torch.float16)
    M, K = x.shape
    N = codes.shape[0]
    _need(codes, "codes", torch.uint8, (N, K // 2))
    _need(scales, "scales", torch.uint8, (N, K // 16))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, "out", torch.float32, (M, N))
    _check("qgemm_nvfp4_w4a16", lib().qgemm_nvfp4_w4a16(codes.data_ptr(), scales.data_ptr(), float(global_scale),
                                                        x.data_ptr(), out.data_ptr(), M, N, K, _stream(stream)))
    return out


def _group_outs(x, Ns, outs):
    M = x.shape[0]
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.float32, device=x.device) for n in Ns]
    for i, o in enumerate(outs):
        _need(o, f"out[{i}]", torch.float32, (M, Ns[i]))
    return outs


def qgemm_nvfp4_w4a16_group(codes, scales, global_scales, x: torch.Tensor, outs=None, stream=None):
    """Several NVFP4 matrices reading the same x in one launch; returns the outputs."""
    count = len(codes)
    if not 1 <= count <= 8 or len(scales) != count or len(global_scales) != count:
        raise ValueError("need 1..8 matrices with their scales and global scales")
    _need(x, "x", torch.float16)
    M, K = x.shape
    Ns = [c.shape[0] for c in codes]
    for i in range(count):
        _need(codes[i], f"codes[{i}]", torch.uint8, (Ns[i], K // 2))
        _need(scales[i], f"scales[{i}]", torch.uint8, (Ns[i], K // 16))
    outs = _group_outs(x, Ns, outs)
    arr = ctypes.c_void_p * count
    cp, sp, yp = arr(*[c.data_ptr() for c in codes]), arr(*[t.data_ptr() for t in scales]), arr(*[o.data_ptr() for o in outs])
    gp = (ctypes.c_float * count)(*[float(g) for g in global_scales])
    npa = (ctypes.c_int64 * count)(*Ns)
    _check("qgemm_nvfp4_w4a16_group", lib().qgemm_nvfp4_w4a16_group(count, cp, sp, gp, x.data_ptr(), yp, npa, M, K,
                                                                    _stream(stream)))
    return outs


def qgemm_fp8_w8a16_group(ws, row_scales, x: torch.Tensor, outs=None, stream=None):
    """Several FP8 matrices reading the same x in one launch; returns the outputs."""
    count = len(ws)
    if not 1 <= count <= 8 or len(row_scales) != count:
        raise ValueError("need 1..8 matrices with their row scales")
    _need(x, "x", torch.float16)
    M, K = x.shape
    Ns = [w.shape[0] for w in ws]
    for i in range(count):
        _need(ws[i], f"w[{i}]", torch.uint8, (Ns[i], K))
        _need(row_scales[i], f"row_scale[{i}]", torch.float32, (Ns[i],))
    outs = _group_outs(x, Ns, outs)
    arr = ctypes.c_void_p * count
    wp, rp, yp = arr(*[w.data_ptr() for w in ws]), arr(*[r.data_ptr() for r in row_scales]), arr(*[o.data_ptr() for o in outs])
    npa = (ctypes.c_int64 * count)(*Ns)
    _check("qgemm_fp8_w8a16_group", lib().qgemm_fp8_w8a16_group(count, wp, rp, x.data_ptr(), yp, npa, M, K,
                                                                _stream(stream)))
    return outs


def qgemm_fp8_w8a16(w: torch.Tensor, row_scale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """FP8 E4M3 uint8 [N, K], fp32 row scale [N], x fp16 [M, K] -> fp32 [M, N]."""
    _need(x, "x", torch.float16)
    M, K = x.shape
    N = w.shape[0]
    _need(w, "w", torch.uint8, (N, K))
    _need(row_scale, "row_scale", torch.float32, (N,))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, "out", torch.float32, (M, N))
    _check("qgemm_fp8_w8a16", lib().qgemm_fp8_w8a16(w.data_ptr(), row_scale.data_ptr(), x.data_ptr(),
                                                    out.data_ptr(), M, N, K, _stream(stream)))
    return out


def set_launch_overlap(enable: bool) -> None:
    """Programmatic dependent launch between consecutive calls (see qmv.h)."""
    lib().qmv_set_launch_overlap(int(bool(enable)))


def get_launch_overlap() -> bool:
    return bool(lib().qmv_get_launch_overlap())


def route_counts() -> dict:
    L = lib()
    return {L.qmv_route_name(i).decode(): int(L.qmv_route_launches(i)) for i in range(L.qmv_route_count())}


def route_reset() -> None:
    lib().qmv_route_reset()


def error_flags(clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check("qmv_error_flags", lib().qmv_error_flags(ctypes.byref(v), int(clear)))
    return int(v.value)

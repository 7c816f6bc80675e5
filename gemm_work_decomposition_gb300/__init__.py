"""Work-decomposed BF16 GEMM for GB300: Python binding of libsk.so (include/sk.h).

Argument marshalling only: every function forwards to the C entry point of the same
name. Pointers may be given as integers or as objects with `data_ptr()` (torch
tensors); streams as integers (cudaStream_t), objects with `cuda_stream`, or None
(the legacy default stream). Negative return codes raise SkError. The library is
loaded on first use and its absence is an error: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsk.so")

# enums and constants of include/sk.h
SK_DP, SK_SPLITK, SK_STREAMK, SK_HYBRID = 0, 1, 2, 3
SK_NN, SK_NT = 0, 1
SK_DETERMINISTIC, SK_ATOMIC = 0, 1
SK_F32, SK_BF16 = 0, 1
SK_ROLE_FULL, SK_ROLE_OWNER, SK_ROLE_PRODUCER, SK_ROLE_SLAB = 0, 1, 2, 3
SK_OK, SK_EINVAL, SK_EWORKSPACE, SK_ECUDA, SK_ETIMEOUT, SK_ECAPACITY, SK_ERESIDENCY, SK_EBOUNDS = 0, -1, -2, -3, -4, -5, -6, -7
SK_TILE_M, SK_TILE_N, SK_BLK_K = 128, 128, 64
SK_MAP_VERSION, SK_MAP_HEADER, SK_MAP_SEG, SK_MAP_TILE = 3, 18, 9, 4
SK_TILE_128x128, SK_TILE_256x128_PAIR, SK_TILE_256x256_PAIR, SK_TILE_128x256 = 0, 1, 2, 3
SK_WS_HEADER_BYTES = 256
SK_TRACE_SEGS = 15
SK_TRACE_WORDS = 4 + 4 * SK_TRACE_SEGS

EXPORTS = ("sk_plan_size", "sk_plan", "sk_workspace_size", "sk_gemm", "sk_gemm_debug", "sk_reduce_splits",
           "sk_status", "sk_strerror", "sk_gemm_noalloc", "sk_split_k_slices", "sk_host_staging_size",
           "sk_gemm_host")
SK_NOALLOC_SCRATCH_BYTES = 16 << 20


class sk_schedule(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("splits", ctypes.c_int32), ("units", ctypes.c_int32),
                ("min_iters", ctypes.c_int32), ("split_partials", ctypes.c_int32), ("tile", ctypes.c_int32),
                ("raster", ctypes.c_int32), ("swizzle", ctypes.c_int32), ("overlap", ctypes.c_int32),
                ("sk_groups", ctypes.c_int32)]


class sk_debug_opts(ctypes.Structure):
    _fields_ = [("reverse_units", ctypes.c_int32), ("skip_producer_signal", ctypes.c_int32),
                ("timeout_ns", ctypes.c_int64), ("dump", ctypes.c_void_p), ("trace", ctypes.c_void_p),
                ("zero_partials", ctypes.c_int32)]


class SkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {sk_strerror(code)} ({code})")


def schedule(mode: int, splits: int = 1, units: int = 0, min_iters: int = 0, split_partials: int = 0,
             tile: int = 0, raster: int = 0, swizzle: int = 0, overlap: int = 0, sk_groups: int = 0) -> sk_schedule:
    return sk_schedule(mode, splits, units, min_iters, split_partials, tile, raster, swizzle, overlap, sk_groups)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libsk.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with gemm_work_decomposition_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        L.sk_plan_size.argtypes = [i32, i32, i32, i32, sk_schedule]
        L.sk_plan_size.restype = i64
        L.sk_plan.argtypes = [i32, i32, i32, i32, sk_schedule, ctypes.POINTER(i32), i64]
        L.sk_plan.restype = i32
        L.sk_workspace_size.argtypes = [i32, i32, i32, i32, sk_schedule, i32]
        L.sk_workspace_size.restype = i64
        gemm_args = [vp, vp, vp, i32, i32, i32, i32, i32, sk_schedule, i32, i32, vp, sz, vp]
        L.sk_gemm.argtypes = gemm_args
        L.sk_gemm.restype = i32
        L.sk_gemm_debug.argtypes = gemm_args + [ctypes.POINTER(sk_debug_opts)]
        L.sk_gemm_debug.restype = i32
        L.sk_reduce_splits.argtypes = [vp, vp, i32, i32, i64, vp]
        L.sk_reduce_splits.restype = i32
        L.sk_status.argtypes = [vp, vp]
        L.sk_status.restype = i32
        L.sk_gemm_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, sk_schedule, i32, i32, vp]
        L.sk_gemm_noalloc.restype = i32
        L.sk_split_k_slices.argtypes = [i32, i32, i32, i32]
        L.sk_split_k_slices.restype = i32
        L.sk_host_staging_size.argtypes = [i32, i32, i32, i32, i32]
        L.sk_host_staging_size.restype = i64
        L.sk_gemm_host.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), i32, i32, i32,
                                   i32, i32, sk_schedule, i32, i32, vp, sz, i32, vp, sz, vp, vp, vp]
        L.sk_gemm_host.restype = i32
        L.sk_strerror.argtypes = [i32]
        L.sk_strerror.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(code: int, where: str) -> int:
    if code < 0:
        raise SkError(int(code), where)
    return code


def sk_strerror(code: int) -> str:
    return lib().sk_strerror(code).decode()


def sk_plan_size(M: int, N: int, K: int, num_sms: int, sched: sk_schedule) -> int:
    return _check(lib().sk_plan_size(M, N, K, num_sms, sched), "sk_plan_size")


def sk_plan(M: int, N: int, K: int, num_sms: int, sched: sk_schedule) -> np.ndarray:
    """The work-unit map as an int32 array (layout in include/sk.h)."""
    n = sk_plan_size(M, N, K, num_sms, sched)
    out = np.zeros(n, dtype=np.int32)
    _check(lib().sk_plan(M, N, K, num_sms, sched, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n), "sk_plan")
    return out


def sk_split_k_slices(M: int, N: int, K: int, num_sms: int) -> int:
    """The CUTLASS page's Split-K factor for this problem (include/sk.h)."""
    return _check(lib().sk_split_k_slices(M, N, K, num_sms), "sk_split_k_slices")


def sk_workspace_size(M: int, N: int, K: int, num_sms: int, sched: sk_schedule, reduction: int) -> int:
    return _check(lib().sk_workspace_size(M, N, K, num_sms, sched, reduction), "sk_workspace_size")


def sk_gemm(A, B, C, c_dtype: int, M: int, N: int, K: int, layout: int, sched: sk_schedule, reduction: int,
            num_sms: int, workspace, ws_bytes: int, stream=None) -> int:
    return _check(lib().sk_gemm(_ptr(A), _ptr(B), _ptr(C), c_dtype, M, N, K, layout, sched, reduction, num_sms,
                                _ptr(workspace), ws_bytes, _stream(stream)), "sk_gemm")


def sk_gemm_debug(A, B, C, c_dtype: int, M: int, N: int, K: int, layout: int, sched: sk_schedule, reduction: int,
                  num_sms: int, workspace, ws_bytes: int, stream=None, reverse_units: int = 0,
                  skip_producer_signal: int = 0, timeout_ns: int = 0, dump=None, trace=None,
                  zero_partials: int = 0) -> int:
    opts = sk_debug_opts(reverse_units, skip_producer_signal, timeout_ns, _ptr(dump) or None, _ptr(trace) or None,
                         zero_partials)
    return _check(lib().sk_gemm_debug(_ptr(A), _ptr(B), _ptr(C), c_dtype, M, N, K, layout, sched, reduction,
                                      num_sms, _ptr(workspace), ws_bytes, _stream(stream), ctypes.byref(opts)),
                  "sk_gemm_debug")


def sk_reduce_splits(P, C, c_dtype: int, splits: int, mn: int, stream=None) -> int:
    return _check(lib().sk_reduce_splits(_ptr(P), _ptr(C), c_dtype, splits, mn, _stream(stream)), "sk_reduce_splits")


def sk_status(workspace, stream=None) -> int:
    """Device status word (SK_OK or SK_ETIMEOUT), read and reset. Raises only on SK_ECUDA."""
    code = lib().sk_status(_ptr(workspace), _stream(stream))
    if code in (SK_ECUDA, SK_EWORKSPACE):
        raise SkError(code, "sk_status")
    return code


def sk_gemm_noalloc(A, B, C, c_dtype: int, M: int, N: int, K: int, layout: int, sched: sk_schedule, reduction: int,
                    num_sms: int, stream=None) -> int:
    """sk_gemm on the library-owned scratch (no workspace argument); see include/sk.h."""
    return _check(lib().sk_gemm_noalloc(_ptr(A), _ptr(B), _ptr(C), c_dtype, M, N, K, layout, sched, reduction,
                                        num_sms, _stream(stream)), "sk_gemm_noalloc")


def sk_host_staging_size(M: int, N: int, K: int, c_dtype: int, depth: int) -> int:
    return _check(lib().sk_host_staging_size(M, N, K, c_dtype, depth), "sk_host_staging_size")


def sk_gemm_host(A, B, C, c_dtype: int, M: int, N: int, K: int, layout: int, sched: sk_schedule, reduction: int,
                 num_sms: int, staging, staging_bytes: int, depth: int, workspace, ws_bytes: int, stream=None,
                 copy_in=None, copy_out=None) -> int:
    """`len(C)` GEMMs over host buffers (sequences of host pointers or CPU tensors, one per
    problem) through the device staging buffer; see include/sk.h."""
    n = len(C)
    if len(A) != n or len(B) != n:
        raise ValueError("A, B and C must hold one buffer per problem")
    arr = ctypes.c_void_p * max(n, 1)
    pa, pb, pc = arr(*[_ptr(x) for x in A]), arr(*[_ptr(x) for x in B]), arr(*[_ptr(x) for x in C])
    return _check(lib().sk_gemm_host(n, pa, pb, pc, c_dtype, M, N, K, layout, sched, reduction, num_sms,
                                     _ptr(staging), staging_bytes, depth, _ptr(workspace), ws_bytes,
                                     _stream(stream), _stream(copy_in), _stream(copy_out)), "sk_gemm_host")

"""CPU oracle for the per-tensor-scaled E4M3 GEMM, HGEMM and E4M3 quantiser.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg import this package; the product library
(``fp16_tensor_core_gb300``) never does, and shares no code with it.

The arithmetic lives in ``dg_oracle.c`` (plain C, FP64 accumulation, tables
built from the number-format definitions).  This module only marshals numpy
arrays into it.  Citations use these page shorthands:

* [FP8-guide] "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南" (sheratonhq.com/news/156926)
* [DG-FP16]   the DeepGEMM FP16/WMMA deep-dive page (hnwysp.cn/news/84236)
* [HGEMM-L2]  "HGEMM优化：深度学习中的矩阵乘法性能提升策略" (jsqmd.com/news/710660)

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(format facts, worked rounding cases, closed forms, an independent integer
formulation, brute force and library cross-checks).
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np

from . import build as _build

_lib = None
_lock = threading.Lock()

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(_build.build())
            L.dgo_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.dgo_e4m3_decode.restype = ctypes.c_double
            L.dgo_e4m3_encode.argtypes = [ctypes.c_double]
            L.dgo_e4m3_encode.restype = ctypes.c_uint8
            L.dgo_fp16_decode.argtypes = [ctypes.c_uint16]
            L.dgo_fp16_decode.restype = ctypes.c_double
            L.dgo_bf16_decode.argtypes = [ctypes.c_uint16]
            L.dgo_bf16_decode.restype = ctypes.c_double
            L.dgo_bf16_encode.argtypes = [ctypes.c_float]
            L.dgo_bf16_encode.restype = ctypes.c_uint16
            L.dgo_fp16_encode.argtypes = [ctypes.c_double]
            L.dgo_fp16_encode.restype = ctypes.c_uint16
            L.dgo_amax.argtypes = [_f32p, _i64]
            L.dgo_amax.restype = ctypes.c_float
            L.dgo_scale_from_amax.argtypes = [ctypes.c_float]
            L.dgo_scale_from_amax.restype = ctypes.c_float
            L.dgo_scale_pow2_from_amax.argtypes = [ctypes.c_float]
            L.dgo_scale_pow2_from_amax.restype = ctypes.c_float
            L.dgo_fp16_range_scale.argtypes = [ctypes.c_float, ctypes.c_float, _f32p]
            L.dgo_fp16_range_scale.restype = None
            L.dgo_convert_f16.argtypes = [_f32p, _i64, ctypes.c_float, _u16p]
            L.dgo_convert_f16.restype = None
            L.dgo_quantize_e4m3.argtypes = [_f32p, _i64, ctypes.c_float, _u8p]
            L.dgo_quantize_e4m3.restype = None
            L.dgo_gemm_e4m3.argtypes = [_u8p, _u8p, _i64, _i64, _i64, _f64p,
                                        ctypes.c_void_p, ctypes.c_int]
            L.dgo_gemm_e4m3.restype = None
            L.dgo_hgemm.argtypes = [_u16p, _u16p, _i64, _i64, _i64, _f64p,
                                    ctypes.c_void_p, ctypes.c_int]
            L.dgo_hgemm.restype = None
            L.dgo_gemm_e4m3_at.argtypes = [_u8p, _u8p, _i64, _i64p, _i64p, _i64,
                                           _f64p, ctypes.c_void_p]
            L.dgo_gemm_e4m3_at.restype = None
            L.dgo_hgemm_at.argtypes = [_u16p, _u16p, _i64, _i64p, _i64p, _i64,
                                       _f64p, ctypes.c_void_p]
            L.dgo_hgemm_at.restype = None
            L.dgo_epilogue_scale.argtypes = [_f64p, _i64, ctypes.c_float,
                                             ctypes.c_float, _f64p]
            L.dgo_epilogue_scale.restype = None
            L.dgo_epilogue_e4m3.argtypes = [_f64p, _i64, ctypes.c_float,
                                            ctypes.c_float, ctypes.c_float, _u8p]
            L.dgo_epilogue_e4m3.restype = None
            L.dgo_gemm_e4m3_exact_i64.argtypes = [_u8p, _u8p, _i64, _i64, _i64, _i64p]
            L.dgo_gemm_e4m3_exact_i64.restype = ctypes.c_int
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr_or_none(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# -- number formats ---------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3 codes to float64 ([FP8-guide] §2.1, §4.3)."""
    L = lib()
    tab = np.array([L.dgo_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return tab[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(values) -> np.ndarray:
    """Nearest-even, saturating E4M3 encode of float64 values ([FP8-guide] §4.3)."""
    L = lib()
    v = np.asarray(values, dtype=np.float64)
    out = np.fromiter((L.dgo_e4m3_encode(float(x)) for x in v.ravel()),
                      dtype=np.uint8, count=v.size)
    return out.reshape(v.shape)


def fp16_decode(bits) -> np.ndarray:
    L = lib()
    tab = np.array([L.dgo_fp16_decode(h) for h in range(65536)], dtype=np.float64)
    return tab[np.asarray(bits, dtype=np.uint16)]


def bf16_decode(bits) -> np.ndarray:
    L = lib()
    b = np.asarray(bits, dtype=np.uint16)
    tab = np.array([L.dgo_bf16_decode(h) for h in range(65536)], dtype=np.float64)
    return tab[b]


def bf16_encode(values) -> np.ndarray:
    L = lib()
    v = np.asarray(values, dtype=np.float32)
    out = np.fromiter((L.dgo_bf16_encode(float(x)) for x in v.ravel()),
                      dtype=np.uint16, count=v.size)
    return out.reshape(v.shape)


def fp16_encode(values) -> np.ndarray:
    L = lib()
    v = np.asarray(values, dtype=np.float64)
    out = np.fromiter((L.dgo_fp16_encode(float(x)) for x in v.ravel()),
                      dtype=np.uint16, count=v.size)
    return out.reshape(v.shape)


# -- per-tensor scaling and the quantiser -----------------------------------

def amax(x) -> np.float32:
    """max |x_i|, NaN-propagating ([FP8-guide] §3.2)."""
    x = _c(x, np.float32).ravel()
    return np.float32(lib().dgo_amax(x, x.size))


def scale_from_amax(a) -> np.float32:
    """fl32(amax / 448), 1 for amax == 0 ([FP8-guide] §3.2)."""
    return np.float32(lib().dgo_scale_from_amax(float(np.float32(a))))


def scale_pow2_from_amax(a) -> np.float32:
    """Smallest power of two p with 448 p >= amax ([FP8-guide] §2.1)."""
    return np.float32(lib().dgo_scale_pow2_from_amax(float(np.float32(a))))


def quantize_tensor_pow2(x):
    """(codes, scale, amax) with the power-of-two per-tensor scale."""
    a = amax(x)
    s = scale_pow2_from_amax(a)
    return quantize_e4m3(x, s), s, a


def fp16_range_scale(amax_a, amax_b) -> np.ndarray:
    """[scale, sqrt(scale), 1/scale, 1] as float32, scale = min(1,
    65504 / (amax_a * amax_b)) ([DG-FP16] §3.3)."""
    out = np.zeros(4, dtype=np.float32)
    lib().dgo_fp16_range_scale(float(np.float32(amax_a)), float(np.float32(amax_b)), out)
    return out


def convert_f16(x, factor) -> np.ndarray:
    """fp16_rn(fl32(x * factor)) elementwise, as uint16 bit patterns."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().dgo_convert_f16(x.ravel(), x.size, float(np.float32(factor)), out.reshape(-1))
    return out


def fp16_range_chain(A32, B32):
    """The whole [DG-FP16] §3.3 path in the oracle: factors, the scaled FP16
    operands and the exact FP64 product of those operands divided by scale.
    Returns (factors, A16, B16, D) with D = R / scale (FP64)."""
    f = fp16_range_scale(amax(A32), amax(B32))
    A16 = convert_f16(A32, f[1])
    B16 = convert_f16(B32, f[1])
    R, S = hgemm(A16, B16)
    return f, A16, B16, R * float(f[2]), S


def quantize_e4m3(x, scale) -> np.ndarray:
    """e4m3(fl32(x / scale)) elementwise ([FP8-guide] §4.3)."""
    x = _c(x, np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    lib().dgo_quantize_e4m3(x.ravel(), x.size, float(np.float32(scale)), q.reshape(-1))
    return q


def quantize_tensor(x):
    """(codes, scale, amax) for one tensor: the page's per-tensor recipe."""
    a = amax(x)
    s = scale_from_amax(a)
    return quantize_e4m3(x, s), s, a


# -- contractions -------------------------------------------------------------

def gemm_e4m3(A, B, with_abs=True, nthreads=0):
    """R = A @ B^T over decoded E4M3 codes in FP64 (and S = sum |a*b|)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    R = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_abs else None
    lib().dgo_gemm_e4m3(A.reshape(-1) if A.size else np.zeros(1, np.uint8),
                        B.reshape(-1) if B.size else np.zeros(1, np.uint8),
                        M, N, K, R.reshape(-1) if R.size else np.zeros(1),
                        _ptr_or_none(S), nthreads)
    return (R, S) if with_abs else R


def hgemm(A, B, with_abs=True, nthreads=0):
    """R = A @ B^T over decoded binary16 bit patterns in FP64 (and S)."""
    A = _c(A, np.uint16)
    B = _c(B, np.uint16)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    R = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_abs else None
    lib().dgo_hgemm(A.reshape(-1) if A.size else np.zeros(1, np.uint16),
                    B.reshape(-1) if B.size else np.zeros(1, np.uint16),
                    M, N, K, R.reshape(-1) if R.size else np.zeros(1),
                    _ptr_or_none(S), nthreads)
    return (R, S) if with_abs else R


def gemm_e4m3_at(A, B, ms, ns):
    """(R, S) of the E4M3 contraction at the selected (m, n) positions."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    R = np.empty(ms.size, dtype=np.float64)
    S = np.empty(ms.size, dtype=np.float64)
    lib().dgo_gemm_e4m3_at(A.reshape(-1), B.reshape(-1), A.shape[1], ms, ns,
                           ms.size, R, _ptr_or_none(S))
    return R, S


def hgemm_at(A, B, ms, ns):
    A = _c(A, np.uint16)
    B = _c(B, np.uint16)
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    R = np.empty(ms.size, dtype=np.float64)
    S = np.empty(ms.size, dtype=np.float64)
    lib().dgo_hgemm_at(A.reshape(-1), B.reshape(-1), A.shape[1], ms, ns,
                       ms.size, R, _ptr_or_none(S))
    return R, S


def epilogue_scale(R, sA, sB) -> np.ndarray:
    """Dref = R * sA * sB in FP64 ([FP8-guide] §3.2)."""
    R = _c(R, np.float64)
    out = np.empty(R.shape, dtype=np.float64)
    if R.size:
        lib().dgo_epilogue_scale(R.reshape(-1), R.size, float(sA), float(sB),
                                 out.reshape(-1))
    return out


def epilogue_e4m3(R, sA, sB, sD) -> np.ndarray:
    """e4m3(R * sA * sB / sD), one rounding ([FP8-guide] §3.2, §4.3)."""
    R = _c(R, np.float64)
    out = np.empty(R.shape, dtype=np.uint8)
    if R.size:
        lib().dgo_epilogue_e4m3(R.reshape(-1), R.size, float(sA), float(sB),
                                float(sD), out.reshape(-1))
    return out


def gemm_e4m3_exact_units(A, B) -> np.ndarray:
    """Independent integer contraction in units of 2^-18 (pins gemm_e4m3)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N = B.shape[0]
    out = np.empty((M, N), dtype=np.int64)
    rc = lib().dgo_gemm_e4m3_exact_i64(A.reshape(-1), B.reshape(-1), M, N, K,
                                       out.reshape(-1))
    if rc != 0:
        raise ValueError("NaN code in input")
    return out

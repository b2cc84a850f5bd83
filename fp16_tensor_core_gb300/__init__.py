"""Python binding of libdg (include/dg.h): argument marshalling only.

Every function below has the name of the C entry point it calls and does no
arithmetic of its own: it turns torch tensors (device memory) into pointers
and sizes, calls the library, and raises DgError on a non-zero status.
PyTorch is used only for device memory and streams.  There is no fallback:
if ``_build/libdg.so`` has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "DG_OK", "DG_ERR_INVALID_VALUE", "DG_ERR_MISALIGNED", "DG_ERR_UNSUPPORTED",
    "DG_ERR_CUDA", "DG_ERR_TIMEOUT", "DG_BF16", "DG_E4M3", "DG_FP16", "DgError",
    "lib", "library_path", "dg_amax", "dg_amax_pow2", "dg_quantize_e4m3",
    "dg_quantize_e4m3_amax", "dg_fp8_gemm",
    "dg_fp8_gemm_amax", "dg_fp8_gemm_grouped", "dg_fp8_gemm_splitk_static",
    "dg_hgemm", "dg_hgemm_scaled", "dg_fp16_range_scale", "dg_convert_f16",
    "dg_gemm_plan", "dg_init", "dg_sync_status", "dg_set_wait_timeout_us",
    "dg_debug_skip_first_load", "dg_status_string", "dg_version", "dg_release_stream",
    "dg_reload_env", "dg_convert_f16_amax", "dg_convert_f16_amax_pair", "dg_quantize_e4m3_pair",
    "EXPORTED_SYMBOLS",
]

DG_OK, DG_ERR_INVALID_VALUE, DG_ERR_MISALIGNED, DG_ERR_UNSUPPORTED, DG_ERR_CUDA, DG_ERR_TIMEOUT = range(6)
DG_BF16, DG_E4M3, DG_FP16 = 0, 1, 2

#: Every function include/dg.h declares.
EXPORTED_SYMBOLS = (
    "dg_amax", "dg_amax_pow2", "dg_quantize_e4m3", "dg_quantize_e4m3_amax", "dg_fp8_gemm",
    "dg_fp8_gemm_amax",
    "dg_fp8_gemm_grouped", "dg_fp8_gemm_splitk_static", "dg_hgemm", "dg_hgemm_scaled",
    "dg_fp16_range_scale", "dg_convert_f16", "dg_gemm_plan",
    "dg_init", "dg_sync_status", "dg_set_wait_timeout_us", "dg_debug_skip_first_load",
    "dg_status_string", "dg_version", "dg_release_stream", "dg_reload_env", "dg_convert_f16_amax",
    "dg_convert_f16_amax_pair", "dg_quantize_e4m3_pair",
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libdg.so")
_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


class DgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dg_status_string(status)} ({status})")


class _Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("path", "block_m", "block_n", "block_k", "stages", "grid", "tiles", "smem_bytes")]


def lib():
    """The loaded libdg (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"libdg.so not found at {_LIB_PATH}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(_LIB_PATH)
            vp, i64, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.dg_amax.argtypes = [vp, i64, vp, vp, vp]
            L.dg_amax_pow2.argtypes = [vp, i64, vp, vp, vp]
            L.dg_quantize_e4m3.argtypes = [vp, i64, vp, vp, vp]
            L.dg_quantize_e4m3_amax.argtypes = [vp, i64, vp, vp, vp, vp, vp]
            L.dg_fp8_gemm.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, ctypes.c_int, vp]
            L.dg_fp8_gemm_amax.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, ctypes.c_int,
                                           vp, vp]
            L.dg_fp8_gemm_grouped.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, vp, vp, vp,
                                              vp, ctypes.c_int, vp]
            L.dg_fp8_gemm_splitk_static.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp,
                                                     ctypes.c_int, vp, vp]
            L.dg_hgemm.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, vp]
            L.dg_hgemm_scaled.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, ctypes.c_int, vp]
            L.dg_fp16_range_scale.argtypes = [vp, vp, vp, vp]
            L.dg_convert_f16.argtypes = [vp, i64, vp, vp, vp]
            L.dg_convert_f16_amax.argtypes = [vp, i64, vp, vp, vp, vp]
            L.dg_convert_f16_amax_pair.argtypes = [vp, i64, vp, i64, vp, vp, vp, vp, vp, vp]
            L.dg_quantize_e4m3_pair.argtypes = [vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp]
            L.dg_gemm_plan.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(_Plan)]
            L.dg_init.argtypes = []
            L.dg_sync_status.argtypes = [vp]
            L.dg_set_wait_timeout_us.argtypes = [ctypes.c_uint64]
            L.dg_set_wait_timeout_us.restype = None
            L.dg_debug_skip_first_load.argtypes = [ctypes.c_int]
            L.dg_debug_skip_first_load.restype = None
            L.dg_status_string.argtypes = [ctypes.c_int]
            L.dg_status_string.restype = ctypes.c_char_p
            L.dg_version.argtypes = []
            L.dg_release_stream.argtypes = [vp]
            L.dg_reload_env.argtypes = []
            L.dg_reload_env.restype = None
            for name in ("dg_amax", "dg_amax_pow2", "dg_quantize_e4m3", "dg_fp8_gemm", "dg_fp8_gemm_amax", "dg_hgemm",
                         "dg_fp8_gemm_grouped", "dg_fp8_gemm_splitk_static", "dg_gemm_plan", "dg_init",
                         "dg_sync_status", "dg_version", "dg_hgemm_scaled", "dg_fp16_range_scale",
                         "dg_convert_f16", "dg_quantize_e4m3_amax", "dg_release_stream",
                         "dg_convert_f16_amax", "dg_convert_f16_amax_pair",
                         "dg_quantize_e4m3_pair"):
                getattr(L, name).restype = st
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor must be in CUDA device memory")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != DG_OK:
        raise DgError(rc, where)


def dg_status_string(status: int) -> str:
    return lib().dg_status_string(int(status)).decode()


def dg_version() -> int:
    return lib().dg_version()


def dg_init() -> None:
    _check(lib().dg_init(), "dg_init")


def dg_amax(x, amax_out, scale_out=None, stream=None) -> None:
    """amax_out[0] = max |x|; scale_out[0] = amax / 448 (1 if amax == 0)."""
    _check(lib().dg_amax(_ptr(x), x.numel(), _ptr(amax_out), _ptr(scale_out), _stream(stream)),
           "dg_amax")


def dg_amax_pow2(x, amax_out, scale_out, stream=None) -> None:
    """amax_out[0] = max |x|; scale_out[0] = smallest power of two p with 448 p >= amax."""
    _check(lib().dg_amax_pow2(_ptr(x), x.numel(), _ptr(amax_out), _ptr(scale_out), _stream(stream)),
           "dg_amax_pow2")


def dg_quantize_e4m3(x, scale, q, stream=None) -> None:
    """q = E4M3(x / scale[0]) elementwise (uint8 codes)."""
    if q.numel() != x.numel():
        raise ValueError("q must have as many elements as x")
    _check(lib().dg_quantize_e4m3(_ptr(x), x.numel(), _ptr(scale), _ptr(q), _stream(stream)),
           "dg_quantize_e4m3")


def dg_quantize_e4m3_pair(a, b, amax_a, amax_b, scale_a, scale_b, qa, qb, stream=None) -> None:
    """amax, scale and E4M3 codes of both GEMM operands in one call (as
    dg_amax + dg_quantize_e4m3 on each)."""
    _check(lib().dg_quantize_e4m3_pair(_ptr(a), a.numel(), _ptr(b), b.numel(), _ptr(amax_a),
                                       _ptr(amax_b), _ptr(scale_a), _ptr(scale_b), _ptr(qa),
                                       _ptr(qb), _stream(stream)), "dg_quantize_e4m3_pair")


def dg_quantize_e4m3_amax(x, scale, q, amax_out, next_scale_out=None, stream=None) -> None:
    """q = E4M3(x / scale[0]) and amax_out[0] = max |x| in one pass; optionally
    next_scale_out[0] = amax / 448 (delayed scaling)."""
    _check(lib().dg_quantize_e4m3_amax(_ptr(x), x.numel(), _ptr(scale), _ptr(q), _ptr(amax_out),
                                       _ptr(next_scale_out), _stream(stream)),
           "dg_quantize_e4m3_amax")


def dg_fp8_gemm(A, B, D, scale_a, scale_b, scale_d=None, out=DG_BF16, stream=None,
                M=None, N=None, K=None) -> None:
    """D (M x N) = out(scale_a * scale_b * A (M x K, E4M3) @ B (N x K, E4M3)^T)."""
    if M is None:
        M, K = A.shape
        N = B.shape[0]
    _check(lib().dg_fp8_gemm(_ptr(A), _ptr(B), _ptr(D), M, N, K, _ptr(scale_a), _ptr(scale_b),
                             _ptr(scale_d), int(out), _stream(stream)), "dg_fp8_gemm")


def dg_fp8_gemm_amax(A, B, D, scale_a, scale_b, scale_d=None, out=DG_BF16, amax_d=None,
                     stream=None, M=None, N=None, K=None) -> None:
    """dg_fp8_gemm, and amax_d[0] = max |scale_a * scale_b * acc| (delayed output scaling)."""
    if M is None:
        M, K = A.shape
        N = B.shape[0]
    _check(lib().dg_fp8_gemm_amax(_ptr(A), _ptr(B), _ptr(D), M, N, K, _ptr(scale_a), _ptr(scale_b),
                                  _ptr(scale_d), int(out), _ptr(amax_d), _stream(stream)),
           "dg_fp8_gemm_amax")


def dg_fp8_gemm_splitk_static(A, B, D, scale_a, scale_b, scale_d=None, out=DG_BF16,
                              status_out=None, stream=None, M=None, N=None, K=None) -> None:
    """dg_fp8_gemm for M <= 16 on the split-K kernel with the library's static
    workspace (no allocation); kernel error bits are ORed into status_out."""
    if M is None:
        M, K = A.shape
        N = B.shape[0]
    _check(lib().dg_fp8_gemm_splitk_static(_ptr(A), _ptr(B), _ptr(D), M, N, K, _ptr(scale_a),
                                           _ptr(scale_b), _ptr(scale_d), int(out),
                                           _ptr(status_out), _stream(stream)),
           "dg_fp8_gemm_splitk_static")


def dg_fp8_gemm_grouped(A, B, D, group_offsets, scale_a, scale_b, scale_d=None, out=DG_BF16,
                        stream=None, M=None, N=None, K=None, groups=None) -> None:
    """Grouped GEMM: group g computes rows [off[g], off[g+1]) of D from B rows [g*N, g*N + N)."""
    if groups is None:
        groups = group_offsets.numel() - 1
    if M is None:
        M, K = A.shape
        N = D.shape[1]
    _check(lib().dg_fp8_gemm_grouped(_ptr(A), _ptr(B), _ptr(D), M, N, K, int(groups),
                                     _ptr(group_offsets), _ptr(scale_a), _ptr(scale_b),
                                     _ptr(scale_d), int(out), _stream(stream)),
           "dg_fp8_gemm_grouped")


def dg_hgemm(A, B, D, out=DG_FP16, stream=None, M=None, N=None, K=None) -> None:
    """D (M x N) = out(A (M x K, FP16) @ B (N x K, FP16)^T), FP32 accumulation."""
    if M is None:
        M, K = A.shape
        N = B.shape[0]
    _check(lib().dg_hgemm(_ptr(A), _ptr(B), _ptr(D), M, N, K, int(out), _stream(stream)),
           "dg_hgemm")


def dg_hgemm_scaled(A, B, D, scale_a, scale_b, out=DG_BF16, stream=None, M=None, N=None,
                    K=None) -> None:
    """D = out(scale_a * scale_b * A @ B^T), FP16 operands, FP32 accumulation."""
    if M is None:
        M, K = A.shape
        N = B.shape[0]
    _check(lib().dg_hgemm_scaled(_ptr(A), _ptr(B), _ptr(D), M, N, K, _ptr(scale_a),
                                 _ptr(scale_b), int(out), _stream(stream)), "dg_hgemm_scaled")


def dg_fp16_range_scale(amax_a, amax_b, factors, stream=None) -> None:
    """factors[0..3] = scale, sqrt(scale), 1/scale, 1 with
    scale = min(1, 65504 / (amax_a * amax_b)) (FP16 dynamic-range scaling)."""
    _check(lib().dg_fp16_range_scale(_ptr(amax_a), _ptr(amax_b), _ptr(factors),
                                     _stream(stream)), "dg_fp16_range_scale")


def dg_convert_f16(x, out, factor=None, stream=None) -> None:
    """out = fp16_rn(x * factor[0]) elementwise (binary16 bit patterns)."""
    _check(lib().dg_convert_f16(_ptr(x), x.numel(), _ptr(factor), _ptr(out), _stream(stream)),
           "dg_convert_f16")


def dg_convert_f16_amax(x, out, factor, amax_out, stream=None) -> None:
    """out = fp16_rn(x * factor[0]) and amax_out[0] = max |x| in one pass
    (the next call's factors come from dg_fp16_range_scale on such maxima)."""
    _check(lib().dg_convert_f16_amax(_ptr(x), x.numel(), _ptr(factor), _ptr(out), _ptr(amax_out),
                                     _stream(stream)), "dg_convert_f16_amax")


def dg_convert_f16_amax_pair(a, b, out_a, out_b, factor, amax_a, amax_b, stream=None) -> None:
    """dg_convert_f16_amax for both HGEMM operands in one pass (one factor)."""
    _check(lib().dg_convert_f16_amax_pair(_ptr(a), a.numel(), _ptr(b), b.numel(), _ptr(factor),
                                          _ptr(out_a), _ptr(out_b), _ptr(amax_a), _ptr(amax_b),
                                          _stream(stream)), "dg_convert_f16_amax_pair")


def dg_gemm_plan(M, N, K, in_dtype=DG_E4M3, out_dtype=DG_BF16, sm_count=0) -> dict:
    """The path and tile the library picks for this shape (host only)."""
    p = _Plan()
    _check(lib().dg_gemm_plan(M, N, K, int(in_dtype), int(out_dtype), int(sm_count),
                              ctypes.byref(p)), "dg_gemm_plan")
    return {f: getattr(p, f) for f, _ in _Plan._fields_}


def dg_sync_status(stream=None) -> int:
    """Synchronise the stream; return (without raising) the status code."""
    return lib().dg_sync_status(_stream(stream))


def dg_set_wait_timeout_us(us: int) -> None:
    lib().dg_set_wait_timeout_us(int(us))


def dg_debug_skip_first_load(enable: bool = True) -> None:
    lib().dg_debug_skip_first_load(1 if enable else 0)


def dg_release_stream(stream=None) -> None:
    """Free the split-K workspace the stream holds (synchronises the stream)."""
    _check(lib().dg_release_stream(_stream(stream)), "dg_release_stream")


def dg_reload_env() -> None:
    """Re-read the DG_* tuning variables (otherwise read once, at first use)."""
    lib().dg_reload_env()

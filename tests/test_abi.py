"""Host-side checks of the C ABI: the library builds, loads and exports every
function include/dg.h declares, argument errors come back as status codes
before anything touches a device, and the tile table behaves.  CPU only: no
call here reaches a kernel launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import fp16_tensor_core_gb300 as dg
from _knobs import knobs
from fp16_tensor_core_gb300 import build as dg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg.h")


@pytest.fixture(scope="module")
def L():
    dg_build.build()
    return dg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(dg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    # and nothing from the oracle leaks into the product library
    with pytest.raises(AttributeError):
        getattr(L, "dgo_gemm_e4m3")


def test_reload_env_reads_the_tuning_variables(L):
    """Tuning variables are read once; a change shows only after dg_reload_env."""
    dg.dg_reload_env()
    assert dg.dg_gemm_plan(16, 12288, 4096, sm_count=152)["path"] == 4
    os.environ["DG_SPLITK"] = "0"
    try:
        assert dg.dg_gemm_plan(16, 12288, 4096, sm_count=152)["path"] == 4   # not re-read yet
        dg.dg_reload_env()
        assert dg.dg_gemm_plan(16, 12288, 4096, sm_count=152)["path"] == 3
    finally:
        os.environ.pop("DG_SPLITK", None)
        dg.dg_reload_env()
    assert dg.dg_gemm_plan(16, 12288, 4096, sm_count=152)["path"] == 4


def test_status_strings_and_version(L):
    assert dg.dg_status_string(dg.DG_OK) == "DG_OK"
    assert dg.dg_status_string(dg.DG_ERR_TIMEOUT) == "DG_ERR_TIMEOUT"
    assert dg.dg_status_string(99) == "DG_ERR_UNKNOWN"
    assert dg.dg_version() >= 100


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced: every call below fails validation


@pytest.mark.parametrize("args,expect", [
    # negative sizes
    ((FAKE, FAKE, FAKE, -1, 8, 16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_INVALID_VALUE),
    ((FAKE, FAKE, FAKE, 8, 8, -16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_INVALID_VALUE),
    # too large
    ((FAKE, FAKE, FAKE, 1 << 31, 8, 16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_INVALID_VALUE),
    # null operands / scales / output
    ((None, FAKE, FAKE, 8, 8, 16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_INVALID_VALUE),
    ((FAKE, FAKE, None, 8, 8, 16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_INVALID_VALUE),
    ((FAKE, FAKE, FAKE, 8, 8, 16, None, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_INVALID_VALUE),
    # E4M3 output needs an output scale
    ((FAKE, FAKE, FAKE, 8, 8, 16, FAKE, FAKE, None, dg.DG_E4M3, None), dg.DG_ERR_INVALID_VALUE),
    # unknown output type
    ((FAKE, FAKE, FAKE, 8, 8, 16, FAKE, FAKE, None, 7, None), dg.DG_ERR_INVALID_VALUE),
    # misaligned pointers or row pitch
    ((FAKE + 1, FAKE, FAKE, 8, 8, 16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_MISALIGNED),
    ((FAKE, FAKE + 8, FAKE, 8, 8, 16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE + 2, 8, 8, 16, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, 8, 8, 24, FAKE, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_MISALIGNED),
    # FP32 scales that a 4-byte load cannot read
    ((FAKE, FAKE, FAKE, 8, 8, 16, FAKE + 1, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, 8, 8, 16, FAKE, FAKE + 2, None, dg.DG_BF16, None), dg.DG_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, 8, 8, 16, FAKE, FAKE, FAKE + 3, dg.DG_E4M3, None), dg.DG_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, 1, 8, 16, FAKE + 1, FAKE, None, dg.DG_BF16, None), dg.DG_ERR_MISALIGNED),
])
def test_fp8_gemm_argument_errors(L, args, expect):
    assert L.dg_fp8_gemm(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((FAKE, FAKE, FAKE, 8, 8, 16, dg.DG_E4M3, None), dg.DG_ERR_INVALID_VALUE),  # bad out type
    ((FAKE, FAKE, FAKE, 8, -1, 16, dg.DG_FP16, None), dg.DG_ERR_INVALID_VALUE),
    ((None, FAKE, FAKE, 8, 8, 16, dg.DG_FP16, None), dg.DG_ERR_INVALID_VALUE),
    ((FAKE, FAKE, FAKE, 8, 8, 12, dg.DG_FP16, None), dg.DG_ERR_MISALIGNED),   # K*2 % 16 != 0
    ((FAKE, FAKE, FAKE + 4, 8, 8, 16, dg.DG_FP16, None), dg.DG_ERR_MISALIGNED),
])
def test_hgemm_argument_errors(L, args, expect):
    assert L.dg_hgemm(*args) == expect


def test_gemm_amax_argument_errors(L):
    ok = (FAKE, FAKE, FAKE, 8, 8, 16, FAKE, FAKE, None, dg.DG_BF16)
    assert L.dg_fp8_gemm_amax(*ok, None, None) == dg.DG_ERR_INVALID_VALUE       # no amax_d
    assert L.dg_fp8_gemm_amax(*ok, FAKE + 2, None) == dg.DG_ERR_MISALIGNED      # amax_d
    bad = (FAKE, FAKE, FAKE, 8, 8, 24, FAKE, FAKE, None, dg.DG_BF16)
    assert L.dg_fp8_gemm_amax(*bad, FAKE, None) == dg.DG_ERR_MISALIGNED        # K pitch
    e4 = (FAKE, FAKE, FAKE, 8, 8, 16, FAKE, FAKE, None, dg.DG_E4M3)
    assert L.dg_fp8_gemm_amax(*e4, FAKE, None) == dg.DG_ERR_INVALID_VALUE      # no scale_d
    sa1 = (FAKE, FAKE, FAKE, 8, 8, 16, FAKE + 1, FAKE, None, dg.DG_BF16)
    assert L.dg_fp8_gemm_amax(*sa1, FAKE, None) == dg.DG_ERR_MISALIGNED        # scale_a


def test_grouped_argument_errors(L):
    base = dict(A=FAKE, B=FAKE, D=FAKE, M=64, N=32, K=16, G=4, off=FAKE, sa=FAKE, sb=FAKE, sd=None,
                out=dg.DG_BF16)

    def call(**kw):
        a = dict(base, **kw)
        return L.dg_fp8_gemm_grouped(a["A"], a["B"], a["D"], a["M"], a["N"], a["K"], a["G"],
                                     a["off"], a["sa"], a["sb"], a["sd"], a["out"], None)
    assert call(G=0) == dg.DG_ERR_INVALID_VALUE
    assert call(G=1025) == dg.DG_ERR_INVALID_VALUE
    assert call(off=None) == dg.DG_ERR_INVALID_VALUE
    assert call(off=FAKE + 2) == dg.DG_ERR_MISALIGNED
    assert call(sa=None) == dg.DG_ERR_INVALID_VALUE
    assert call(out=dg.DG_E4M3) == dg.DG_ERR_INVALID_VALUE      # scale_d missing
    assert call(K=24) == dg.DG_ERR_MISALIGNED
    assert call(M=-1) == dg.DG_ERR_INVALID_VALUE
    assert call(N=1 << 30, G=8) == dg.DG_ERR_INVALID_VALUE      # groups * N overflows
    assert call(sa=FAKE + 1) == dg.DG_ERR_MISALIGNED
    assert call(sb=FAKE + 2) == dg.DG_ERR_MISALIGNED
    assert call(sd=FAKE + 3, out=dg.DG_E4M3) == dg.DG_ERR_MISALIGNED


def test_splitk_static_argument_errors(L):
    """The no-allocation split-K entry rejects what its fixed workspace cannot
    hold, and every other bad argument as dg_fp8_gemm does, before any CUDA
    call."""
    def call(A=FAKE, B=FAKE, D=FAKE, M=8, N=256, K=64, sa=FAKE, sb=FAKE, sd=None,
             out=dg.DG_BF16, status=None):
        return L.dg_fp8_gemm_splitk_static(A, B, D, M, N, K, sa, sb, sd, out, status, None)
    assert call(M=17) == dg.DG_ERR_INVALID_VALUE                 # more rows than the MMA's 16
    assert call(N=128 * 1024 + 1) == dg.DG_ERR_INVALID_VALUE     # more than 1024 tiles
    assert call(M=-1) == dg.DG_ERR_INVALID_VALUE
    assert call(out=7) == dg.DG_ERR_INVALID_VALUE
    assert call(out=dg.DG_E4M3) == dg.DG_ERR_INVALID_VALUE       # scale_d missing
    assert call(sa=None) == dg.DG_ERR_INVALID_VALUE
    assert call(D=None) == dg.DG_ERR_INVALID_VALUE
    assert call(K=24) == dg.DG_ERR_MISALIGNED
    assert call(A=FAKE + 8) == dg.DG_ERR_MISALIGNED
    assert call(status=FAKE + 2) == dg.DG_ERR_MISALIGNED
    assert call(sa=FAKE + 1) == dg.DG_ERR_MISALIGNED
    assert call(sb=FAKE + 2) == dg.DG_ERR_MISALIGNED
    assert call(sd=FAKE + 3, out=dg.DG_E4M3) == dg.DG_ERR_MISALIGNED
    assert call(M=0) == dg.DG_OK and call(N=0) == dg.DG_OK       # empty: nothing launched


def test_fp16_range_argument_errors(L):
    assert L.dg_fp16_range_scale(None, FAKE, FAKE, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_fp16_range_scale(FAKE, FAKE, None, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_fp16_range_scale(FAKE + 2, FAKE, FAKE, None) == dg.DG_ERR_MISALIGNED
    assert L.dg_fp16_range_scale(FAKE, FAKE, FAKE + 4, None) == dg.DG_ERR_MISALIGNED  # 16 B
    assert L.dg_convert_f16(FAKE, -1, None, FAKE, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_convert_f16(None, 8, None, FAKE, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_convert_f16(FAKE + 4, 8, None, FAKE, None) == dg.DG_ERR_MISALIGNED
    assert L.dg_convert_f16(FAKE, 8, None, FAKE + 8, None) == dg.DG_ERR_MISALIGNED
    assert L.dg_convert_f16(FAKE, 8, FAKE + 1, FAKE, None) == dg.DG_ERR_MISALIGNED
    h = (FAKE, FAKE, FAKE, 8, 8, 16)
    assert L.dg_hgemm_scaled(*h, None, FAKE, dg.DG_BF16, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_hgemm_scaled(*h, FAKE, FAKE, dg.DG_E4M3, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_hgemm_scaled(*h, FAKE + 2, FAKE, dg.DG_BF16, None) == dg.DG_ERR_MISALIGNED
    assert L.dg_hgemm_scaled(FAKE, FAKE, FAKE, 8, 8, 12, FAKE, FAKE, dg.DG_BF16,
                             None) == dg.DG_ERR_MISALIGNED


def test_convert_f16_amax_argument_errors(L):
    c = L.dg_convert_f16_amax
    assert c(FAKE, -1, None, FAKE, FAKE + 64, None) == dg.DG_ERR_INVALID_VALUE
    assert c(FAKE, 8, None, FAKE, None, None) == dg.DG_ERR_INVALID_VALUE        # no amax word
    assert c(None, 8, None, FAKE, FAKE, None) == dg.DG_ERR_INVALID_VALUE
    assert c(FAKE, 8, FAKE + 64, FAKE, FAKE + 64, None) == dg.DG_ERR_INVALID_VALUE   # amax is factor
    assert c(FAKE + 4, 8, None, FAKE, FAKE, None) == dg.DG_ERR_MISALIGNED
    assert c(FAKE, 8, None, FAKE + 8, FAKE, None) == dg.DG_ERR_MISALIGNED
    assert c(FAKE, 8, FAKE + 1, FAKE, FAKE + 64, None) == dg.DG_ERR_MISALIGNED
    assert c(FAKE, 8, None, FAKE, FAKE + 2, None) == dg.DG_ERR_MISALIGNED


def test_convert_f16_amax_pair_argument_errors(L):
    c = L.dg_convert_f16_amax_pair
    A, B, F, OA, OB, MA, MB = FAKE, FAKE + 256, FAKE + 512, FAKE + 768, FAKE + 1024, FAKE + 1280, FAKE + 1296
    assert c(A, -1, B, 8, None, OA, OB, MA, MB, None) == dg.DG_ERR_INVALID_VALUE
    assert c(A, 8, B, -1, None, OA, OB, MA, MB, None) == dg.DG_ERR_INVALID_VALUE
    assert c(A, 8, B, 8, None, OA, OB, None, MB, None) == dg.DG_ERR_INVALID_VALUE      # no amax word
    assert c(A, 8, B, 8, None, OA, OB, MA, None, None) == dg.DG_ERR_INVALID_VALUE
    assert c(None, 8, B, 8, None, OA, OB, MA, MB, None) == dg.DG_ERR_INVALID_VALUE
    assert c(A, 8, B, 8, None, OA, None, MA, MB, None) == dg.DG_ERR_INVALID_VALUE
    assert c(A, 8, B, 8, None, OA, OB, MA, MA, None) == dg.DG_ERR_INVALID_VALUE      # one word for both
    assert c(A, 8, B, 8, F, OA, OB, F, MB, None) == dg.DG_ERR_INVALID_VALUE          # amax is factor
    assert c(A, 8, B, 8, F, OA, OB, MA, F, None) == dg.DG_ERR_INVALID_VALUE
    assert c(A + 4, 8, B, 8, None, OA, OB, MA, MB, None) == dg.DG_ERR_MISALIGNED
    assert c(A, 8, B + 4, 8, None, OA, OB, MA, MB, None) == dg.DG_ERR_MISALIGNED
    assert c(A, 8, B, 8, None, OA, OB + 8, MA, MB, None) == dg.DG_ERR_MISALIGNED
    assert c(A, 8, B, 8, F + 1, OA, OB, MA, MB, None) == dg.DG_ERR_MISALIGNED
    assert c(A, 8, B, 8, None, OA, OB, MA, MB + 2, None) == dg.DG_ERR_MISALIGNED


def test_quantize_pair_argument_errors(L):
    q = L.dg_quantize_e4m3_pair
    A, B, QA, QB = FAKE, FAKE + 256, FAKE + 512, FAKE + 768
    W = [FAKE + 1024 + 16 * i for i in range(4)]
    assert q(A, -1, B, 8, *W, QA, QB, None) == dg.DG_ERR_INVALID_VALUE
    assert q(A, 8, B, -1, *W, QA, QB, None) == dg.DG_ERR_INVALID_VALUE
    for k in range(4):                                       # each word required
        w = list(W)
        w[k] = None
        assert q(A, 8, B, 8, *w, QA, QB, None) == dg.DG_ERR_INVALID_VALUE
    assert q(None, 8, B, 8, *W, QA, QB, None) == dg.DG_ERR_INVALID_VALUE
    assert q(A, 8, B, 8, *W, QA, None, None) == dg.DG_ERR_INVALID_VALUE
    for i in range(4):                                       # the four words distinct
        for j in range(i + 1, 4):
            w = list(W)
            w[j] = w[i]
            assert q(A, 8, B, 8, *w, QA, QB, None) == dg.DG_ERR_INVALID_VALUE, (i, j)
    assert q(A + 4, 8, B, 8, *W, QA, QB, None) == dg.DG_ERR_MISALIGNED
    assert q(A, 8, B, 8, *W, QA, QB + 4, None) == dg.DG_ERR_MISALIGNED
    assert q(A, 8, B, 8, W[0] + 2, *W[1:], QA, QB, None) == dg.DG_ERR_MISALIGNED


def test_quantize_amax_argument_errors(L):
    q = L.dg_quantize_e4m3_amax
    assert q(FAKE, 10, None, FAKE, FAKE, None, None) == dg.DG_ERR_INVALID_VALUE    # no scale
    assert q(FAKE, 10, FAKE, FAKE, None, None, None) == dg.DG_ERR_INVALID_VALUE    # no amax
    assert q(FAKE, -1, FAKE, FAKE, FAKE + 64, None, None) == dg.DG_ERR_INVALID_VALUE
    assert q(FAKE, 10, FAKE, FAKE, FAKE, None, None) == dg.DG_ERR_INVALID_VALUE    # amax is scale
    assert q(FAKE + 4, 10, FAKE, FAKE, FAKE + 64, None, None) == dg.DG_ERR_MISALIGNED
    assert q(FAKE, 10, FAKE, FAKE, FAKE + 66, None, None) == dg.DG_ERR_MISALIGNED
    assert q(FAKE, 10, FAKE, FAKE, FAKE + 64, FAKE + 1, None) == dg.DG_ERR_MISALIGNED


def test_moe_group_sizes_recipe():
    import synth
    s = synth.moe_group_sizes(3, 16, 8192, empty=2)
    assert s.sum() == 8192 and (s[:2] == 0).all() and (s[2:] > 0).all()
    assert s.max() > 4 * max(1, int(np.median(s[2:])))   # skewed load
    A, B, off = synth.make_moe_inputs(4, 300, 32, 64, empty=1)
    assert A.shape == (300, 64) and B.shape == (128, 64) and off[0] == 0 and off[-1] == 300


def test_scale_and_quantise_argument_errors(L):
    assert L.dg_amax(FAKE, -1, FAKE, None, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_amax(FAKE, 10, None, None, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_amax(None, 10, FAKE, None, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_amax(FAKE + 4, 10, FAKE, None, None) == dg.DG_ERR_MISALIGNED
    assert L.dg_amax(FAKE, 10, FAKE + 2, None, None) == dg.DG_ERR_MISALIGNED
    assert L.dg_amax_pow2(FAKE, 10, FAKE, None, None) == dg.DG_ERR_INVALID_VALUE  # scale required
    assert L.dg_amax_pow2(FAKE + 8, 10, FAKE, FAKE, None) == dg.DG_ERR_MISALIGNED
    assert L.dg_quantize_e4m3(FAKE, 10, None, FAKE, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_quantize_e4m3(FAKE, -3, FAKE, FAKE, None) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_quantize_e4m3(FAKE, 10, FAKE, FAKE + 1, None) == dg.DG_ERR_MISALIGNED


def test_plan_decode_shapes_default_to_warp_mma(L):
    """1 <= M <= 16: the warp-MMA GEMV (path 5) except where it measured
    slower -- E4M3 with 9-16 rows of A against a large N * K (split-K), and
    M = 1 E4M3 beyond one wave of 4-warp CTAs (CUDA-core GEMV)."""
    sm = 152
    for m, n, k, fp16, path, warps in (
            (1, 12288, 4096, False, 5, 4),     # 768 CTAs: one wave of 4-warp CTAs
            (8, 12288, 4096, False, 5, 4),
            (2, 28672, 4096, False, 5, 2),     # 1792 CTAs: several waves
            (1, 28672, 4096, False, 2, None),  # M = 1 E4M3 there: the CUDA-core GEMV
            (4, 4096, 4096, False, 5, 8),      # 256 CTAs: at most two per SM
            (16, 1000, 1040, False, 5, 8),     # small N * K
            (9, 12288, 4096, False, 4, None),  # 9-16 rows, large N * K: split-K
            (16, 12288, 4096, False, 4, None),
            (16, 12288, 4096, True, 5, 2),     # FP16 operands
            (1, 12288, 4096, True, 5, 4)):
        p = dg.dg_gemm_plan(m, n, k, dg.DG_FP16 if fp16 else dg.DG_E4M3,
                            dg.DG_FP16 if fp16 else dg.DG_BF16, sm_count=sm)
        assert p["path"] == path, (m, n, k, fp16, p)
        if path == 5:
            assert p["block_n"] == 16 and p["grid"] == (n + 15) // 16 and p["tiles"] == p["grid"]
            assert p["block_m"] == (8 if m <= 8 else 16) and p["stages"] == warps, p
    with knobs(DG_MMA_GEMV="1"):
        assert dg.dg_gemm_plan(16, 12288, 4096, sm_count=sm)["path"] == 5
        assert dg.dg_gemm_plan(17, 12288, 4096, sm_count=sm)["path"] != 5
    with knobs(DG_MMA_GEMV_WARPS="3"):
        assert dg.dg_gemm_plan(4, 12288, 4096, sm_count=sm)["stages"] == 3
    # a K longer than the path's 32-bit byte offsets: not path 5
    assert dg.dg_gemm_plan(4, 64, (1 << 31) - 16, sm_count=sm)["path"] != 5


def test_plan_paths_and_tiles(L):
    """The CUDA-core GEMV, split-K and tiled choices, with the warp-MMA GEMV
    and split-K row ranges turned off (the kernels stay selectable and are
    tested on their own)."""
    with knobs(DG_MMA_GEMV="0", DG_SPLITK_ROWS="0"):
        _plan_paths_and_tiles(152)


def test_plan_splitk_row_ranges(L):
    """With DG_SPLITK_ROWS=1, split-K plans with N within 128 rows per SM
    take row ranges: ceil(N / SMs) rows of B per CTA over the whole of K, one
    CTA per range (grid = tiles); wider N keeps 128-row tiles, and so does
    every plan by default."""
    sm = 152
    with knobs(DG_MMA_GEMV="0", DG_SPLITK_ROWS="1"):
        for m, n, rows, tiles in ((16, 12288, 81, 152), (3, 12288, 81, 152), (16, 4096, 27, 152),
                                  (5, 1000, 7, 143), (3, 17, 1, 17), (16, 19456, 128, 152)):
            p = dg.dg_gemm_plan(m, n, 4096, sm_count=sm)
            assert p["path"] == 4 and p["block_n"] == rows, (m, n, p)
            assert p["tiles"] == tiles and p["grid"] == tiles, (m, n, p)
            assert (tiles - 1) * rows < n <= tiles * rows
        p = dg.dg_gemm_plan(16, 19457, 4096, sm_count=sm)   # 129 rows per SM: 128-row tiles
        assert p["path"] == 4 and p["block_n"] == 128 and p["tiles"] == 153
        p = dg.dg_gemm_plan(64, 4096, 4096, sm_count=sm)
        assert p["path"] == 4 and p["block_m"] == 64 and p["block_n"] == 27
        assert p["grid"] == p["tiles"] == 152
    # the decode default at M = 9..16 (E4M3, large N x K): 128-row split-K tiles
    p = dg.dg_gemm_plan(16, 12288, 4096, sm_count=sm)
    assert p["path"] == 4 and p["block_n"] == 128 and p["tiles"] == 96


def _plan_paths_and_tiles(sm):
    assert dg.dg_gemm_plan(0, 10, 16, sm_count=sm)["path"] == 0
    assert dg.dg_gemm_plan(10, 0, 16, sm_count=sm)["path"] == 0
    assert dg.dg_gemm_plan(10, 10, 0, sm_count=sm)["path"] == 1
    # M <= 2, rows of B <= 8 KB: the fewest rows per CTA whose grid fits in one
    # wave of 8 CTAs per SM; if none fits, 8 (E4M3) or 4 (FP16)
    for m in (1, 2):
        for n, rows in ((12288, 16), (4096, 4), (1000, 4), (28672, 8)):
            p = dg.dg_gemm_plan(m, n, 4096, sm_count=sm)
            assert p["path"] == 2 and p["block_n"] == rows and p["grid"] == (n + rows - 1) // rows, (m, n, p)
    assert dg.dg_gemm_plan(1, 4096, 14336, sm_count=sm)["block_n"] == 8     # 14 KB rows
    # the layout's own residency decides: 4 rows x 3 chunks (6 CTAs per SM)
    # while it fits one wave, then 4 x 2 (8 per SM); M = 2 has only 4 x 2 (6)
    p = dg.dg_gemm_plan(1, 12288, 4096, sm_count=sm)
    assert (p["block_n"], p["stages"]) == (16, 3)
    p = dg.dg_gemm_plan(1, 16384, 4096, sm_count=sm)
    assert (p["block_n"], p["stages"]) == (16, 2)
    assert dg.dg_gemm_plan(2, 16384, 4096, sm_count=sm)["block_n"] == 8
    assert dg.dg_gemm_plan(1, 4096, 4096, sm_count=sm)["stages"] == 8
    for n, rows in ((12288, 16), (4096, 4), (28672, 4)):
        p = dg.dg_gemm_plan(1, n, 4096, in_dtype=dg.DG_FP16, out_dtype=dg.DG_FP16, sm_count=sm)
        assert p["path"] == 2 and p["block_n"] == rows, (n, p)
    for m in (3, 16):
        # split-K: 96 tiles of 128 rows of B, 96 x 32 K blocks over 152 CTAs
        p = dg.dg_gemm_plan(m, 12288, 4096, sm_count=sm)
        assert p["path"] == 4 and p["block_m"] == 16 and p["block_n"] == 128
        assert p["tiles"] == 96 and p["grid"] == sm and p["block_k"] == 128
        assert p["smem_bytes"] <= 232448
    # few tiles: a whole multiple of the tile count (every CTA one segment)
    assert dg.dg_gemm_plan(16, 4096, 4096, sm_count=sm)["grid"] == 128    # 4 x 32 tiles
    assert dg.dg_gemm_plan(16, 2048, 4096, sm_count=sm)["grid"] == 144    # 9 x 16 tiles
    assert dg.dg_gemm_plan(16, 11008, 4096, sm_count=sm)["grid"] == sm    # 86 tiles: every SM
    # fewer K blocks than SMs: one per CTA
    p = dg.dg_gemm_plan(5, 200, 256, sm_count=sm)
    assert p["path"] == 4 and p["tiles"] == 2 and p["grid"] == 4
    assert dg.dg_gemm_plan(5, 200, 256, in_dtype=dg.DG_FP16, out_dtype=dg.DG_FP16,
                           sm_count=sm)["grid"] == 8
    os.environ["DG_SPLITK"] = "0"
    dg.dg_reload_env()
    try:
        assert dg.dg_gemm_plan(3, 12288, 4096, sm_count=sm)["path"] == 3
    finally:
        del os.environ["DG_SPLITK"]
        dg.dg_reload_env()
    # 17 <= M <= 128: split-K only where the tiled plan leaves SMs idle and the
    # time estimate favours it (few columns of A, or a long K per tile)
    for m in (17, 32):
        p = dg.dg_gemm_plan(m, 4096, 4096, sm_count=sm)
        assert p["path"] == 4 and p["block_m"] == 32 and p["stages"] == 5
    for m in (48, 64):
        p = dg.dg_gemm_plan(m, 4096, 4096, sm_count=sm)
        assert p["path"] == 4 and p["block_m"] == 64
        assert p["grid"] == 128   # 4 CTAs for each of the 32 tiles
    p = dg.dg_gemm_plan(64, 4096, 11008, sm_count=sm)
    assert p["path"] == 4 and p["block_m"] == 64 and p["stages"] == 4
    p = dg.dg_gemm_plan(64, 4096, 11008, in_dtype=dg.DG_FP16, out_dtype=dg.DG_FP16, sm_count=sm)
    assert p["path"] == 4 and p["block_k"] == 64
    for m, n, k in ((17, 12288, 4096), (128, 4096, 4096),
                    (64, 1024, 4096), (128, 32768, 4096), (129, 4096, 4096)):
        assert dg.dg_gemm_plan(m, n, k, sm_count=sm)["path"] == 3, (m, n, k)
    os.environ["DG_SPLITK"] = "1"
    dg.dg_reload_env()
    try:
        for m, nc in ((33, 64), (64, 64), (65, 128), (128, 128)):
            p = dg.dg_gemm_plan(m, 4096, 4096, sm_count=sm)
            assert p["path"] == 4 and p["block_m"] == nc and p["smem_bytes"] <= 232448
        assert dg.dg_gemm_plan(128, 32768, 4096, sm_count=sm)["path"] == 4
        assert dg.dg_gemm_plan(129, 4096, 4096, sm_count=sm)["path"] == 3
    finally:
        del os.environ["DG_SPLITK"]
        dg.dg_reload_env()
    assert dg.dg_gemm_plan(16, 128 * 8192 + 1, 64, sm_count=sm)["path"] == 3   # too many tiles
    os.environ["DG_GEMV_MAX_M"] = "16"
    dg.dg_reload_env()
    try:
        for m, rows in ((4, 8), (5, 4), (16, 4)):
            p = dg.dg_gemm_plan(m, 12288, 4096, sm_count=sm)
            assert p["path"] == 2 and p["block_n"] == rows and p["grid"] == 12288 // rows
    finally:
        del os.environ["DG_GEMV_MAX_M"]
        dg.dg_reload_env()
    for m in (17, 63, 65, 129, 256, 4096, 8192):
        p = dg.dg_gemm_plan(m, 1000, 1040, sm_count=sm)
        assert p["path"] == 3
        assert p["block_n"] in (64, 96, 128, 160, 192, 224, 256)
        if p["block_m"] == 256:            # CTA pairs: M >= 256, even grid
            assert m >= 256 and p["grid"] % 2 == 0 and p["grid"] <= 2 * p["tiles"]
        else:
            assert p["block_m"] == 128 and p["grid"] <= p["tiles"]
        assert p["grid"] <= sm
        assert p["smem_bytes"] <= 232448
        assert p["block_k"] == 128
    # decode batches on the QKV shape: 128 tiles of 128 x 96 keep 128 SMs
    # streaming B (128 x 128 tiles would keep 96)
    for m in (32, 64, 128):
        p = dg.dg_gemm_plan(m, 12288, 4096, sm_count=sm)
        assert (p["path"], p["block_m"], p["block_n"], p["tiles"], p["grid"]) == (3, 128, 96, 128, 128)
        # two 128-byte K blocks per stage from 12 K blocks on (3 stages)
        assert (p["block_k"], p["stages"]) == (256, 3), p
    p = dg.dg_gemm_plan(129, 1000, 1040, sm_count=sm)   # 9 K blocks: one per stage
    assert (p["block_n"], p["block_k"]) == (64, 128), p
    # the boundary: 11 K blocks one per stage, 12 two (FP16: 64-element blocks)
    assert dg.dg_gemm_plan(32, 12288, 1408, sm_count=sm)["block_k"] == 128
    assert dg.dg_gemm_plan(32, 12288, 1536, sm_count=sm)["block_k"] == 256
    assert dg.dg_gemm_plan(32, 12288, 704, dg.DG_FP16, dg.DG_BF16, sm_count=sm)["block_k"] == 64
    assert dg.dg_gemm_plan(32, 12288, 768, dg.DG_FP16, dg.DG_BF16, sm_count=sm)["block_k"] == 128
    # 9..16 rows over a short K with many tiles: the one-wave tiled kernel;
    # over a long K, or with few tiles, split-K
    p = dg.dg_gemm_plan(16, 12288, 1040, sm_count=sm)
    assert (p["path"], p["block_n"], p["tiles"]) == (3, 96, 128), p
    assert dg.dg_gemm_plan(16, 12288, 4096, sm_count=sm)["path"] == 4
    assert dg.dg_gemm_plan(16, 4096, 1040, sm_count=sm)["path"] == 4
    # the rule's edges: 16 K blocks tiled, 17 split-K; 76 tiles (half the
    # SMs) tiled, 75 split-K
    assert dg.dg_gemm_plan(16, 12288, 2048, sm_count=sm)["path"] == 3
    assert dg.dg_gemm_plan(16, 12288, 2176, sm_count=sm)["path"] == 4
    assert dg.dg_gemm_plan(16, 4864, 1040, sm_count=sm)["path"] == 3
    assert dg.dg_gemm_plan(16, 4800, 1040, sm_count=sm)["path"] == 4
    # CTA pairs: two K blocks per stage from 12 K blocks on (3 stages of 64 KB)
    p = dg.dg_gemm_plan(8192, 8192, 1408, sm_count=sm)
    assert (p["block_m"], p["block_k"], p["stages"]) == (256, 128, 6), p
    p = dg.dg_gemm_plan(8192, 8192, 1536, sm_count=sm)
    assert (p["block_m"], p["block_k"], p["stages"]) == (256, 256, 3), p
    # a 96-wide one-wave plan keeps the tiled kernel over a long K too
    assert dg.dg_gemm_plan(17, 11008, 4096, sm_count=sm)["block_n"] == 96
    # FP16 operands: 64 K elements (128 bytes) per K block; CTA pairs over
    # 4096 K elements (64 K blocks) take two per stage
    p = dg.dg_gemm_plan(4096, 4096, 4096, in_dtype=dg.DG_FP16, out_dtype=dg.DG_FP16, sm_count=sm)
    assert (p["block_m"], p["block_k"]) == (256, 128), p
    p = dg.dg_gemm_plan(4096, 4096, 4096, sm_count=sm)   # E4M3 pairs: 2 x 128 per stage
    assert (p["block_m"], p["block_k"]) == (256, 256), p
    # edge waste: a narrow N problem gets narrower tiles than a wide one
    small = dg.dg_gemm_plan(65, 1000, 1040, sm_count=sm)
    big = dg.dg_gemm_plan(8192, 8192, 8192, sm_count=sm)
    assert small["block_n"] < big["block_n"]
    assert big["grid"] == sm and big["block_m"] == 256 and big["block_n"] == 256
    # 4096^3: 304 pair tiles of 256 x 224, exactly four waves over 76 pairs
    sq = dg.dg_gemm_plan(4096, 4096, 4096, sm_count=sm)
    assert (sq["block_m"], sq["block_n"], sq["tiles"]) == (256, 224, 304)
    with knobs(DG_SPLIT_TAIL="1"):   # with the split tail: 256 tiles of 256 x 256, the
        sq = dg.dg_gemm_plan(4096, 4096, 4096, sm_count=sm)   # last 28 split along K
        assert (sq["block_m"], sq["block_n"], sq["tiles"]) == (256, 256, 256)


def test_plan_argument_errors(L):
    p = dg._Plan()
    assert L.dg_gemm_plan(4, 4, 16, dg.DG_BF16, dg.DG_BF16, 10, ctypes.byref(p)) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_gemm_plan(-4, 4, 16, dg.DG_E4M3, dg.DG_BF16, 10, ctypes.byref(p)) == dg.DG_ERR_INVALID_VALUE
    assert L.dg_gemm_plan(4, 4, 16, dg.DG_E4M3, dg.DG_BF16, 10, None) == dg.DG_ERR_INVALID_VALUE


def test_product_package_does_not_import_oracle():
    """The product path must not route through the CPU oracle."""
    pkg = os.path.join(ROOT, "fp16_tensor_core_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "dg_oracle" not in src, f


def test_plain_c_client_builds_and_runs(L, tmp_path):
    """include/dg.h is valid C and libdg.so links and answers from C."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    exe = tmp_path / "abi_smoke"
    lib_dir = os.path.dirname(dg.library_path())
    src = os.path.join(ROOT, "tests", "c_abi", "abi_smoke.c")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    src, "-o", str(exe), "-L", lib_dir, "-ldg", f"-Wl,-rpath,{lib_dir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "c abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)


def test_tuning_variables_documented():
    """Every DG_* environment variable the library reads is listed in
    include/dg.h, and every one listed there is read."""
    api = open(os.path.join(ROOT, "fp16_tensor_core_gb300", "csrc", "dg_api.cu")).read()
    read = set(re.findall(r'(?:getenv|env_int)\("(DG_[A-Z0-9_]+)"', api))
    header = open(os.path.join(ROOT, "include", "dg.h")).read()
    start = header.index("void dg_reload_env(void);")
    block = header[header.rindex("/*", 0, start):start]
    listed = set(re.findall(r"\b(DG_[A-Z0-9_]+)=", block))
    assert read and read == listed, (sorted(read - listed), sorted(listed - read))

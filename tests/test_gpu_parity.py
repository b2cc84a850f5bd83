"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Every workload of the pages is covered: the 256^3 GEMM, the M in {1, 63, 65,
129} x 1000 x 1040 edge sweep, the decode QKV projection, 4096^3 FP8 and
FP16, and 8192^3 with E4M3 output, each through the full chain FP32 ->
amax -> scale -> quantise -> GEMM -> scaled output.  Every case compares every
output element with the oracle, the full-size 4096^3 and 8192^3 ones too,
in the same launch configuration the benchmark times.
"""
import json
import os

import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import (check_bf16_like, check_e4m3, check_guards, check_quantised, dev,
                     fp16_bits_to_f64, bf16_bits_to_f64, gpu_quantize, guarded,
                     sample_positions, scalar)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def fp8_chain(A32, B32, out=dg.DG_BF16, sd=None, full=True, samples=2048):
    M, K = A32.shape
    N = B32.shape[0]
    qa, amax_a, sa = gpu_quantize(A32)
    qb, amax_b, sb = gpu_quantize(B32)
    qa_ref, sa_ref = check_quantised(A32, qa, amax_a, sa)
    qb_ref, sb_ref = check_quantised(B32, qb, amax_b, sb)
    if out == dg.DG_E4M3:
        buf, D = guarded(M * N, torch.uint8, 0x7F)
        sdt = scalar()
        sdt[0] = float(sd)
    else:
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
        sdt = None
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, sdt, out, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F if out == dg.DG_E4M3 else 0x7FFF)
    h = D.cpu().numpy().reshape(M, N)
    if full:
        if out == dg.DG_E4M3:   # the E4M3 check needs no sum of |a b|
            R, S = oracle.gemm_e4m3(qa_ref, qb_ref, with_abs=False), None
        else:
            R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
        got = h
    else:
        ms, ns = sample_positions(M, N, samples)
        R, S = oracle.gemm_e4m3_at(qa_ref, qb_ref, ms, ns)
        got = h[ms, ns]
    if out == dg.DG_E4M3:
        return check_e4m3(got, R, sa_ref, sb_ref, np.float32(sd))
    d = bf16_bits_to_f64(got.view(np.uint16))
    return check_bf16_like(d, R, S, sa_ref, sb_ref)


# ------------------------------------------------------------- workloads

def test_fp8_256_cubed():
    A, B = synth.make_inputs("fp8_256")
    fp8_chain(A, B)


@pytest.mark.parametrize("name", ["fp8_sweep_m1", "fp8_sweep_m63", "fp8_sweep_m65", "fp8_sweep_m129"])
def test_fp8_edge_sweep(name):
    A, B = synth.make_inputs(name)
    fp8_chain(A, B)


def test_fp8_qkv_decode_projection():
    A, B = synth.make_inputs("fp8_qkv")
    fp8_chain(A, B)


def test_fp8_4096_cubed_all_outputs():
    A, B = synth.make_inputs("fp8_4096")
    fp8_chain(A, B)


@pytest.mark.slow
def test_fp8_8192_cubed_e4m3_out_all_outputs():
    rec = json.load(open(os.path.join(GOLDEN, "sd_8192.json")))
    A, B = synth.make_inputs("fp8_8192_e4m3out")
    fp8_chain(A, B, out=dg.DG_E4M3, sd=rec["scale_d"])


def test_fp8_4096_cubed_sampled_smoke():
    """Quick sampled check (random outputs plus corners) of the same chain."""
    A, B = synth.make_inputs("fp8_4096")
    fp8_chain(A, B, full=False, samples=2000)


def hgemm_case(A16, B16, out=dg.DG_FP16, full=True, samples=2048):
    M, K = A16.shape
    N = B16.shape[0]
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dA, dB = dev(A16.view(np.int16)), dev(B16.view(np.int16))
    dg.dg_hgemm(dA, dB, D, out, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    h = D.cpu().numpy().view(np.uint16).reshape(M, N)
    if full:
        R, S = oracle.hgemm(A16, B16)
        got = h
    else:
        ms, ns = sample_positions(M, N, samples)
        R, S = oracle.hgemm_at(A16, B16, ms, ns)
        got = h[ms, ns]
    d = fp16_bits_to_f64(got) if out == dg.DG_FP16 else bf16_bits_to_f64(got)
    return check_bf16_like(d, R, S, 1.0, 1.0, "FP16" if out == dg.DG_FP16 else "BF16")


def test_fp16_4096_cubed_all_outputs():
    A, B = synth.make_inputs("fp16_4096")
    hgemm_case(A, B)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (129, 1000, 1040), (65, 200, 64), (1, 1000, 1040),
                                   (16, 300, 512), (17, 40, 8)])
def test_fp16_shapes_full(M, N, K):
    A, B = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    hgemm_case(A, B)
    hgemm_case(A, B, out=dg.DG_BF16)


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("M,N,K", [
    (127, 1000, 1040),   # the page's other edge size
    (128, 256, 128),     # exactly one tile, one K block
    (200, 24, 16),       # K smaller than one stage, N < one tile
    (300, 777, 272),     # ragged everywhere, N*2 not a multiple of 16 (scalar stores)
    (2, 1000, 1040),     # warp-MMA GEMV, two rows of A
    (16, 513, 4096),     # warp-MMA GEMV at its M limit
    (17, 64, 64),        # smallest tensor-core M
    (1, 1, 16),          # 1x1 output
    (640, 1536, 2048),   # several waves of tiles over the grid
])
def test_fp8_edge_shapes(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    fp8_chain(A, B)


@pytest.mark.parametrize("M,N,K", [(65, 1000, 1040), (1, 1000, 1040), (256, 256, 256), (300, 777, 272)])
def test_fp8_e4m3_out_small(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, sa, _ = oracle.quantize_tensor(A)
    qb, sb, _ = oracle.quantize_tensor(B)
    R = oracle.gemm_e4m3(qa, qb, with_abs=False)
    sd = np.float32(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))) / 448.0)
    fp8_chain(A, B, out=dg.DG_E4M3, sd=sd)


def test_fp8_fp16_output_type():
    A, B = synth.make_inputs("fp8_sweep_m65", M=130, N=96, K=256)
    qa, amax_a, sa = gpu_quantize(A)
    qb, amax_b, sb = gpu_quantize(B)
    D = torch.empty((130, 96), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_FP16)
    assert dg.dg_sync_status() == dg.DG_OK
    qa_ref, sa_ref = check_quantised(A, qa, amax_a, sa)
    qb_ref, sb_ref = check_quantised(B, qb, amax_b, sb)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(fp16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref, "FP16")


def test_all_ones_gives_k():
    """[FP8-guide] §5.4: all-ones inputs give K in every output."""
    for (M, N, K) in [(1, 64, 4096), (200, 300, 1040)]:
        A = np.ones((M, K), np.float32)
        B = np.ones((N, K), np.float32)
        qa, _, sa = gpu_quantize(A)
        qb, _, sb = gpu_quantize(B)
        D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
        assert dg.dg_sync_status() == dg.DG_OK
        d = D.float().cpu().numpy()
        assert np.all(np.abs(d - K) <= K * 2.0 ** -7), (d.min(), d.max())


def test_k_zero_writes_zeros_and_empty_is_noop():
    D = torch.full((5, 7), 3.0, dtype=torch.bfloat16, device="cuda")
    s = scalar()
    s[0] = 1.0
    A = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((7, 0), dtype=torch.uint8, device="cuda")
    dg.dg_fp8_gemm(A, B, D, s, s, None, dg.DG_BF16, M=5, N=7, K=0)
    assert dg.dg_sync_status() == dg.DG_OK
    assert torch.all(D == 0)
    D2 = torch.full((4,), 3.0, dtype=torch.bfloat16, device="cuda")
    dg.dg_fp8_gemm(A, B, D2, s, s, None, dg.DG_BF16, M=0, N=4, K=16)
    assert torch.all(D2 == 3.0)


# ------------------------------------------------------- amax / quantiser

@pytest.mark.parametrize("n", [0, 1, 3, 4, 5, 511, 512, 513, 4097, 1 << 20, (1 << 20) + 7])
def test_amax_and_quantise_sizes(n):
    x = synth.normal_f32(50 + n % 97, (n,)) * np.float32(3.0)
    q, amax, scale = gpu_quantize(x) if n else (None, None, None)
    if n == 0:
        amax, scale = scalar(), scalar()
        dg.dg_amax(torch.empty(0, dtype=torch.float32, device="cuda"), amax, scale)
        assert dg.dg_sync_status() == dg.DG_OK
        assert amax[0].item() == 0.0 and scale[0].item() == 1.0
        return
    assert dg.dg_sync_status() == dg.DG_OK
    check_quantised(x, q, amax, scale)


def test_amax_special_values():
    base = synth.normal_f32(7, (4099,))
    cases = {
        "zeros": np.zeros(1000, np.float32),
        "negzero": -np.zeros(1000, np.float32),
        "inf": np.concatenate([base, np.float32([-np.inf])]),
        "nan": np.concatenate([base, np.float32([np.nan]), base]),
        "denormal": np.float32([1e-45, -3e-42, 0.0, 1e-40]),
        "huge": np.float32([3.0e38, -3.4e38, 1.0]),
    }
    for name, x in cases.items():
        dx = dev(x)
        amax, scale = scalar(), scalar()
        dg.dg_amax(dx, amax, scale)
        assert dg.dg_sync_status() == dg.DG_OK
        a_ref = oracle.amax(x)
        s_ref = oracle.scale_from_amax(a_ref)
        a, s = amax[0].item(), scale[0].item()
        if np.isnan(a_ref):
            assert np.isnan(a) and np.isnan(s), name
        else:
            assert np.float32(a).view(np.uint32) == np.float32(a_ref).view(np.uint32), name
            assert np.float32(s).view(np.uint32) == np.float32(s_ref).view(np.uint32), name


def _quantise_with(x, s):
    dx = dev(x)
    st = scalar()
    st[0] = float(s)
    q = torch.empty(dx.shape, dtype=torch.uint8, device="cuda")
    dg.dg_quantize_e4m3(dx, st, q)
    assert dg.dg_sync_status() == dg.DG_OK
    return q.cpu().numpy()


def _nan_aware_equal(got, ref):
    nan_ref = (ref & 0x7F) == 0x7F
    nan_got = (got & 0x7F) == 0x7F
    assert np.array_equal(nan_ref, nan_got)
    ok = ~nan_ref
    bad = np.flatnonzero(got[ok] != ref[ok])
    assert bad.size == 0, (bad[:5], got[ok][bad[:5]], ref[ok][bad[:5]])


def test_quantise_special_values_and_scales():
    specials = np.float32([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-45, -1e-45, 1e-38, 3e38,
                           448.0, 464.0, -464.0, 432.0, 2.0 ** -10, 3 * 2.0 ** -10, -(2.0 ** -11)])
    x = np.concatenate([specials, synth.normal_f32(8, (10000,)) * np.float32(100.0)])
    for s in [1.0, 0.37, 3.0e-3, 1.7e4, 2.0 ** -20, 1e-30, 7.0e30]:
        _nan_aware_equal(_quantise_with(x, s), oracle.quantize_e4m3(x, np.float32(s)))


def test_quantise_random_scales_1e7():
    x = synth.normal_f32(77, (10_000_000,)) * np.float32(50.0)
    for s in [0.113, 0.9999999]:
        _nan_aware_equal(_quantise_with(x, s), oracle.quantize_e4m3(x, np.float32(s)))


@pytest.mark.slow
def test_quantise_exhaustive_fp32_scale_one():
    """Every one of the 2^32 binary32 bit patterns at scale = 1."""
    chunk = 1 << 28
    for c in range((1 << 32) // chunk):
        bits = np.arange(chunk, dtype=np.uint32) + np.uint32(c * chunk)
        x = bits.view(np.float32)
        _nan_aware_equal(_quantise_with(x, 1.0), oracle.quantize_e4m3(x, np.float32(1.0)))


# ------------------------------------------------------------- failure path

def test_bounded_wait_reports_timeout_and_context_survives():
    """A pipeline stage that nothing loads: the MMA thread's bounded wait runs
    out, the kernel records DG_ERR_TIMEOUT and returns; the context stays
    usable and the next GEMM is correct."""
    A, B = synth.make_inputs("fp8_256")
    qa, _, sa = gpu_quantize(A)
    qb, _, sb = gpu_quantize(B)
    D = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
    assert dg.dg_sync_status() == dg.DG_OK
    dg.dg_set_wait_timeout_us(100_000)
    try:
        dg.dg_debug_skip_first_load(True)
        dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
        assert dg.dg_sync_status() == dg.DG_ERR_TIMEOUT
        assert dg.dg_sync_status() == dg.DG_OK   # cleared
    finally:
        dg.dg_set_wait_timeout_us(2_000_000)
        dg.dg_debug_skip_first_load(False)
    fp8_chain(A, B)


@pytest.mark.parametrize("M,N,K,rows", [
    (1, 1000, 1040, 4),      # 1 row x 8 chunks per warp
    (2, 4001, 2048, 4),
    (1, 12288, 1024, 16),    # 4 rows x 2 chunks per warp: 768 CTAs, one wave
    (2, 12000, 1040, 16),    # ragged last CTA
    (1, 16000, 512, 16),     # 4 x 3 would not fit one wave: 4 rows x 2 chunks
    (1, 30000, 512, 8),      # no width fits one wave: 2 rows x 4 chunks
])
def test_gemv_one_wave_layouts(M, N, K, rows):
    """M <= 2 on the CUDA-core GEMV (the warp-MMA path turned off): the
    planner's rows per CTA (the fewest whose grid fits one wave) for E4M3 and
    FP16 operands, every element against the oracle."""
    with knobs(DG_MMA_GEMV="0"):
        _gemv_layout_case(M, N, K, rows)


def _gemv_layout_case(M, N, K, rows):
    p = dg.dg_gemm_plan(M, N, K)
    assert p["path"] == 2 and p["block_n"] == rows, p
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    fp8_chain(A, B)
    p16 = dg.dg_gemm_plan(M, N, K, dg.DG_FP16, dg.DG_FP16)
    assert p16["path"] == 2 and p16["block_n"] == (4 if rows == 8 else rows), p16
    A16, B16 = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    hgemm_case(A16, B16)


@pytest.mark.parametrize("M,N,K", [(4, 1000, 1040), (7, 513, 512), (16, 513, 4096), (3, 300, 272)])
def test_gemv_for_larger_m_when_forced(M, N, K):
    """The GEMV handles M up to 16 (its 2-, 4-, 8- and 16-row instantiations),
    although the planner only sends M <= 2 to it by default."""
    os.environ["DG_GEMV_MAX_M"] = "16"
    os.environ["DG_MMA_GEMV"] = "0"
    dg.dg_reload_env()
    try:
        assert dg.dg_gemm_plan(M, N, K)["path"] == 2
        A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
        fp8_chain(A, B)
        A16, B16 = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
        hgemm_case(A16, B16)
    finally:
        del os.environ["DG_GEMV_MAX_M"]
        del os.environ["DG_MMA_GEMV"]
        dg.dg_reload_env()

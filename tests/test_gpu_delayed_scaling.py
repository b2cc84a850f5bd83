"""dg_fp8_gemm_amax: the GEMM also reports max |sA*sB*acc| of its output, and
that value, over 448, serves as the next call's E4M3 output scale (delayed
scaling; [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南" §3.2).

Checked against the oracle's max |Dref| on every kernel path: warp-MMA GEMV
(M <= 8 by default), CUDA-core GEMV and split-K (with the warp-MMA path
off), single CTA, CTA pairs, and FP8 / BF16 outputs.
"""
import os

import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, gpu_quantize, scalar)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def _amax_bound(R, S, sa, sb):
    dref = oracle.epilogue_scale(R, sa, sb)
    i = np.unravel_index(np.argmax(np.abs(dref)), dref.shape)
    ref = float(np.abs(dref[i]))
    # the largest |D| is the maximum of values each within the parity bound
    tol = 8e-3 * ref + 1e-4 * float(np.max(S)) * float(sa) * float(sb)
    return ref, tol


@pytest.mark.parametrize("M,N,K,pairs,path", [
    (1, 1000, 1040, "0", 5),      # warp-MMA GEMV
    (13, 300, 1040, "0", 5),      # warp-MMA GEMV, two MMAs per step
    (1, 1000, 1040, "0", 2),      # CUDA-core GEMV
    (7, 300, 512, "0", 2),        # GEMV, several rows (crossover raised to 16)
    (7, 300, 512, "0", 4),        # the same shape on the split-K kernel
    (16, 1000, 1040, "0", 4),     # split-K, every tile split across CTAs
    (65, 1000, 1040, "0", 4),     # split-K (forced), MMA N = 128
    (65, 1000, 1040, "0", 3),     # single CTA
    (129, 777, 272, "0", 3),      # single CTA, ragged
    (300, 777, 272, "1", 3),      # CTA pairs, odd CTA partly out of range
    (640, 1536, 2048, "1", 3),    # CTA pairs, several tiles per pair
])
def test_output_amax_matches_oracle(M, N, K, pairs, path):
    os.environ["DG_2CTA"] = pairs
    if path in (2, 4):
        os.environ["DG_MMA_GEMV"] = "0"
    dg.dg_reload_env()
    if path == 2:
        os.environ["DG_GEMV_MAX_M"] = "16"
        dg.dg_reload_env()
    if path == 4 and M > 16:
        os.environ["DG_SPLITK"] = "1"
        dg.dg_reload_env()
    try:
        assert dg.dg_gemm_plan(M, N, K, dg.DG_E4M3, dg.DG_BF16)["path"] == path
        A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
        qa, _, sa = gpu_quantize(A)
        qb, _, sb = gpu_quantize(B)
        qa_ref, sa_ref, _ = oracle.quantize_tensor(A)
        qb_ref, sb_ref, _ = oracle.quantize_tensor(B)
        D = torch.empty((M, N), dtype=torch.int16, device="cuda")
        am = scalar()
        am[0] = 123.0   # stale value: the call must reset it
        dg.dg_fp8_gemm_amax(qa, qb, D, sa, sb, None, dg.DG_BF16, am)
        assert dg.dg_sync_status() == dg.DG_OK
        R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
        ref, tol = _amax_bound(R, S, sa_ref, sb_ref)
        got = am[0].item()
        assert abs(got - ref) <= tol, (got, ref, tol)
        # the D written alongside is the ordinary GEMM result
        check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref)
    finally:
        os.environ.pop("DG_2CTA", None)
        os.environ.pop("DG_GEMV_MAX_M", None)
        os.environ.pop("DG_SPLITK", None)
        os.environ.pop("DG_MMA_GEMV", None)
        dg.dg_reload_env()


def test_delayed_scaling_round_trip():
    """Call 1 records amax; call 2 uses sD = amax/448 with E4M3 output: the
    output uses the top of the E4M3 range and matches the oracle within one
    E4M3 step."""
    M, N, K = 384, 1000, 1040
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, _, sa = gpu_quantize(A)
    qb, _, sb = gpu_quantize(B)
    D1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    am = scalar()
    dg.dg_fp8_gemm_amax(qa, qb, D1, sa, sb, None, dg.DG_BF16, am)
    sd = scalar()
    dg.dg_amax(am[0:1].clone(), scalar(), sd)   # sd = amax / 448 via the library's scale rule
    D2 = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    dg.dg_fp8_gemm(qa, qb, D2, sa, sb, sd, dg.DG_E4M3)
    assert dg.dg_sync_status() == dg.DG_OK
    codes = D2.cpu().numpy()
    assert np.max(codes & 0x7F) in (0x7D, 0x7E)      # the largest output lands at ~448
    qa_ref, sa_ref, _ = oracle.quantize_tensor(A)
    qb_ref, sb_ref, _ = oracle.quantize_tensor(B)
    R = oracle.gemm_e4m3(qa_ref, qb_ref, with_abs=False)
    check_e4m3(codes, R, sa_ref, sb_ref, np.float32(sd[0].item()))


def test_empty_and_k_zero_give_zero_amax():
    s = scalar()
    s[0] = 1.0
    am = scalar()
    am[0] = 5.0
    A = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((7, 0), dtype=torch.uint8, device="cuda")
    D = torch.empty((5, 7), dtype=torch.bfloat16, device="cuda")
    dg.dg_fp8_gemm_amax(A, B, D, s, s, None, dg.DG_BF16, am, M=5, N=7, K=0)
    assert dg.dg_sync_status() == dg.DG_OK
    assert am[0].item() == 0.0 and torch.all(D == 0)


@pytest.mark.parametrize("n", [0, 1, 511, 512, 513, 4096 * 5 + 3, 1 << 21])
def test_quantise_with_recorded_scale_and_amax_in_one_pass(n):
    """dg_quantize_e4m3_amax: codes with the given (earlier) scale, this
    tensor's amax and the next scale, all bit-exact against the oracle."""
    x = synth.make_inputs("fp8_sweep_m65", M=1, N=1, K=max(n, 1))[0].reshape(-1)[:n].copy()
    dx = torch.from_numpy(x).cuda() if n else torch.empty(0, dtype=torch.float32, device="cuda")
    scale = scalar()
    scale[0] = 0.0123
    amax, nxt = scalar(), scalar()
    amax[0] = 99.0     # stale: the call must reset it
    q = torch.empty(n, dtype=torch.uint8, device="cuda")
    dg.dg_quantize_e4m3_amax(dx, scale, q, amax, nxt)
    assert dg.dg_sync_status() == dg.DG_OK
    assert np.array_equal(q.cpu().numpy(), oracle.quantize_e4m3(x, np.float32(0.0123)))
    a_ref = oracle.amax(x) if n else np.float32(0.0)
    assert np.float32(amax[0].item()).view(np.uint32) == np.float32(a_ref).view(np.uint32)
    s_ref = oracle.scale_from_amax(a_ref)
    assert np.float32(nxt[0].item()).view(np.uint32) == np.float32(s_ref).view(np.uint32)


def test_quantise_amax_updates_scale_in_place_and_propagates_nan():
    x = synth.normal_f32(21, (100000,))
    scale = scalar()
    scale[0] = 0.01
    amax = scalar()
    q1 = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    dg.dg_quantize_e4m3_amax(torch.from_numpy(x).cuda(), scale, q1, amax, scale)   # next scale in place
    assert dg.dg_sync_status() == dg.DG_OK
    assert np.array_equal(q1.cpu().numpy(), oracle.quantize_e4m3(x, np.float32(0.01)))
    assert scale[0].item() == float(oracle.scale_from_amax(oracle.amax(x)))
    y = x.copy()
    y[777] = np.nan
    dg.dg_quantize_e4m3_amax(torch.from_numpy(y).cuda(), scale, q1, amax)
    assert dg.dg_sync_status() == dg.DG_OK
    assert np.isnan(amax[0].item())

"""The warp-MMA decode GEMV (plan path 5, 1 <= M <= 16) against the oracle.

Forced with DG_MMA_GEMV=1 so that every shape below runs on it whatever the
planner would pick.  Every output is compared: BF16 / FP16 within
8e-3 |Dref| + 1e-4 S sA sB, E4M3 within one step; guard regions around D
catch stores outside [0, M) x [0, N).  Shapes cover both MMA widths (M <= 8
and 9..16), a K tail that is not a whole 64-byte step (and shorter than one
step), N not a multiple of the 16 rows per CTA, both warp counts, FP16
operands, the output-amax report and back-to-back repeatability.
"""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, check_guards, check_quantised,
                     dev, fp16_bits_to_f64, gpu_quantize, guarded, scalar)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    with knobs(DG_MMA_GEMV="1"):
        yield
    assert dg.dg_sync_status() == dg.DG_OK


def _plan(M, N, K, in_dtype=dg.DG_E4M3, out=dg.DG_BF16):
    p = dg.dg_gemm_plan(M, N, K, in_dtype, out)
    assert p["path"] == 5 and p["block_n"] == 16 and p["grid"] == (N + 15) // 16, p
    return p


SHAPES = [
    (1, 1000, 1040),     # M = 1, K tail of 16 bytes past the last whole step
    (2, 4001, 2048),
    (3, 300, 272),
    (8, 12288, 4096),    # the decode QKV weights, one MMA per step
    (9, 513, 512),       # two MMAs per step, ragged N
    (16, 12288, 4096),   # the decode QKV weights, M at the path's limit
    (16, 17, 16),        # K shorter than one 64-byte step, two CTAs, ragged
    (5, 2048, 14336),    # long K
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("warps", ["2", "3", "4", "8"])
def test_fp8_bf16_out(M, N, K, warps):
    with knobs(DG_MMA_GEMV_WARPS=warps):
        assert _plan(M, N, K)["stages"] == int(warps)
        A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
        qa, amax_a, sa = gpu_quantize(A)
        qb, amax_b, sb = gpu_quantize(B)
        qa_ref, sa_ref = check_quantised(A, qa, amax_a, sa)
        qb_ref, sb_ref = check_quantised(B, qb, amax_b, sb)
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
        dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S,
                    sa_ref, sb_ref)


@pytest.mark.parametrize("M,N,K", [(1, 1000, 1040), (12, 3000, 2080)])
def test_fp8_e4m3_and_fp16_out(M, N, K):
    _plan(M, N, K, out=dg.DG_E4M3)
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa_ref, sa, _ = oracle.quantize_tensor(A)
    qb_ref, sb, _ = oracle.quantize_tensor(B)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    sd = np.float32(np.median(np.abs(oracle.epilogue_scale(R, sa, sb))) / 64.0)
    sat, sdt, sbt = scalar(), scalar(), scalar()
    sat[0], sbt[0], sdt[0] = float(sa), float(sb), float(sd)
    buf, D = guarded(M * N, torch.uint8, 0x7F)
    dg.dg_fp8_gemm(dev(qa_ref), dev(qb_ref), D, sat, sbt, sdt, dg.DG_E4M3, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F)
    check_e4m3(D.cpu().numpy().reshape(M, N), R, sa, sb, sd)
    buf16, D16 = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_fp8_gemm(dev(qa_ref), dev(qb_ref), D16, sat, sbt, None, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf16, M * N, 0x7FFF)
    check_bf16_like(fp16_bits_to_f64(D16.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb,
                    "FP16")


@pytest.mark.parametrize("M,N,K", [(1, 1000, 1040), (4, 12288, 4096), (11, 777, 264), (16, 64, 8)])
def test_fp16_operands(M, N, K):
    _plan(M, N, K, dg.DG_FP16, dg.DG_FP16)
    A16, B16 = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A16.view(np.int16)), dev(B16.view(np.int16)), D, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A16, B16)
    check_bf16_like(fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, 1.0, 1.0,
                    "FP16")


def test_output_amax_and_repeatability():
    M, N, K = 13, 2000, 4096
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, _, sa = gpu_quantize(A)
    qb, _, sb = gpu_quantize(B)
    qa_ref, sa_ref, _ = oracle.quantize_tensor(A)
    qb_ref, sb_ref, _ = oracle.quantize_tensor(B)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    am = scalar()
    am[0] = 77.0
    dg.dg_fp8_gemm_amax(qa, qb, D, sa, sb, None, dg.DG_BF16, am)
    assert dg.dg_sync_status() == dg.DG_OK
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    ref = np.max(np.abs(oracle.epilogue_scale(R, sa_ref, sb_ref)))
    i = np.argmax(np.abs(R))
    tol = 8e-3 * ref + 1e-4 * S.reshape(-1)[i] * float(sa_ref) * float(sb_ref)
    assert abs(am[0].item() - ref) <= tol, (am[0].item(), ref, tol)
    outs = [torch.empty_like(D) for _ in range(6)]
    for o in outs:
        dg.dg_fp8_gemm(qa, qb, o, sa, sb, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    for o in outs:
        assert torch.equal(o, D)   # fixed summation order: the same bits every launch

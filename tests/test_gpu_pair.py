"""Parity of the CTA-pair tensor-core kernel (256-row tiles on two SMs) and of
the single-CTA kernel, each selected explicitly, against the CPU oracle.

DG_2CTA=1 / DG_2CTA=0 choose the kernel for every GEMM planned while it is
set; the plan is checked so that each case really runs the kernel it names.
"""
import os

import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, check_guards,
                     check_quantised, dev, fp16_bits_to_f64, gpu_quantize, guarded,
                     scalar)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    os.environ.pop("DG_2CTA", None)
    dg.dg_reload_env()
    assert dg.dg_sync_status() == dg.DG_OK


@pytest.fixture(params=["pair", "single"])
def kernel(request):
    old = os.environ.get("DG_2CTA")
    os.environ["DG_2CTA"] = "1" if request.param == "pair" else "0"
    dg.dg_reload_env()
    yield request.param
    if old is None:
        os.environ.pop("DG_2CTA", None)
        dg.dg_reload_env()
    else:
        os.environ["DG_2CTA"] = old
        dg.dg_reload_env()


def _expect_kernel(kind, M, N, K, in_dtype=dg.DG_E4M3):
    p = dg.dg_gemm_plan(M, N, K, in_dtype, dg.DG_BF16)
    assert p["path"] == 3
    assert p["block_m"] == (256 if kind == "pair" else 128), p


@pytest.mark.parametrize("M,N,K", [
    (256, 256, 256),     # one pair tile row
    (300, 777, 272),     # odd CTA's rows partly out of range, ragged N and K
    (640, 1536, 2048),   # several tiles per pair
    (513, 1000, 1040),   # edge sweep width
    (1024, 4096, 512),   # wide N
])
def test_fp8_bf16_out(kernel, M, N, K):
    _expect_kernel(kernel, M, N, K)
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
    d = bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N))
    check_bf16_like(d, R, S, sa_ref, sb_ref)


_ORACLE_4096 = {}


def test_fp8_4096_all_outputs(kernel):
    """4096^3 on both kernels, every output (the oracle's product is shared
    by the two parametrisations)."""
    _expect_kernel(kernel, 4096, 4096, 4096)
    A, B = synth.make_inputs("fp8_4096")
    qa, amax_a, sa = gpu_quantize(A)
    qb, amax_b, sb = gpu_quantize(B)
    qa_ref, sa_ref = check_quantised(A, qa, amax_a, sa)
    qb_ref, sb_ref = check_quantised(B, qb, amax_b, sb)
    D = torch.empty((4096, 4096), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    if "RS" not in _ORACLE_4096:
        _ORACLE_4096["RS"] = oracle.gemm_e4m3(qa_ref, qb_ref)
    R, S = _ORACLE_4096["RS"]
    d = bf16_bits_to_f64(D.cpu().numpy().view(np.uint16))
    check_bf16_like(d, R, S, sa_ref, sb_ref)


def test_fp8_e4m3_out(kernel):
    M, N, K = 384, 1000, 1040
    _expect_kernel(kernel, M, N, K)
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa_ref, sa, _ = oracle.quantize_tensor(A)
    qb_ref, sb, _ = oracle.quantize_tensor(B)
    R = oracle.gemm_e4m3(qa_ref, qb_ref, with_abs=False)
    sd = np.float32(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))) / 448.0)
    qa, _, sa_d = gpu_quantize(A)
    qb, _, sb_d = gpu_quantize(B)
    sdt = scalar()
    sdt[0] = float(sd)
    buf, D = guarded(M * N, torch.uint8, 0x7F)
    dg.dg_fp8_gemm(qa, qb, D, sa_d, sb_d, sdt, dg.DG_E4M3, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F)
    check_e4m3(D.cpu().numpy().reshape(M, N), R, sa, sb, sd)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (520, 300, 1040)])
def test_fp16_hgemm(kernel, M, N, K):
    _expect_kernel(kernel, M, N, K, dg.DG_FP16)
    A, B = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A.view(np.int16)), dev(B.view(np.int16)), D, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A, B)
    check_bf16_like(fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S,
                    1.0, 1.0, "FP16")


def test_bounded_wait_timeout(kernel):
    """One pipeline stage left unloaded: the bounded wait runs out, the kernel
    reports DG_ERR_TIMEOUT and returns, and the next GEMM is correct."""
    A, B = synth.make_inputs("fp8_256")
    qa, _, sa = gpu_quantize(A)
    qb, _, sb = gpu_quantize(B)
    D = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
    assert dg.dg_sync_status() == dg.DG_OK
    _expect_kernel(kernel, 256, 256, 256)
    dg.dg_set_wait_timeout_us(100_000)
    try:
        dg.dg_debug_skip_first_load(True)
        dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
        assert dg.dg_sync_status() == dg.DG_ERR_TIMEOUT
        assert dg.dg_sync_status() == dg.DG_OK
    finally:
        dg.dg_set_wait_timeout_us(2_000_000)
        dg.dg_debug_skip_first_load(False)
    test_fp8_bf16_out(kernel, 256, 256, 256)


@pytest.mark.parametrize("out", [dg.DG_BF16, dg.DG_FP16, dg.DG_E4M3])
@pytest.mark.parametrize("M,N,K", [(300, 1024, 272), (512, 2048, 128)])
def test_last_tile_bulk_store_epilogue(kernel, M, N, K, out):
    """Rows of D a multiple of 16 bytes: each pair's last tile is written by
    bulk tensor stores (swizzled staging, rows past M clipped); every element
    is checked, and nothing outside D is written."""
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa_ref, sa, _ = oracle.quantize_tensor(A)
    qb_ref, sb, _ = oracle.quantize_tensor(B)
    qa, _, sa_d = gpu_quantize(A)
    qb, _, sb_d = gpu_quantize(B)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    if out == dg.DG_E4M3:
        sd = np.float32(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))) / 448.0)
        sdt = scalar()
        sdt[0] = float(sd)
        buf, D = guarded(M * N, torch.uint8, 0x7F)
        dg.dg_fp8_gemm(qa, qb, D, sa_d, sb_d, sdt, out, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
        check_guards(buf, M * N, 0x7F)
        check_e4m3(D.cpu().numpy().reshape(M, N), R, sa, sb, sd)
    else:
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
        dg.dg_fp8_gemm(qa, qb, D, sa_d, sb_d, None, out, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
        check_guards(buf, M * N, 0x7FFF)
        h = D.cpu().numpy().view(np.uint16).reshape(M, N)
        d = fp16_bits_to_f64(h) if out == dg.DG_FP16 else bf16_bits_to_f64(h)
        check_bf16_like(d, R, S, sa, sb, "FP16" if out == dg.DG_FP16 else "BF16")

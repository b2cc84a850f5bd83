"""Power-of-two per-tensor scales on the GPU (dg_amax_pow2) against the
oracle: bit-exact scale and codes, and the GEMM chain's parity with them.
[FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南" §2.1."""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _parity import bf16_bits_to_f64, check_bf16_like, dev, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def gpu_quantize_pow2(x32):
    dx = dev(x32)
    amax, scale = scalar(), scalar()
    dg.dg_amax_pow2(dx, amax, scale)
    q = torch.empty(dx.shape, dtype=torch.uint8, device="cuda")
    dg.dg_quantize_e4m3(dx, scale, q)
    return q, amax, scale


CASES = {
    "normal": lambda: synth.normal_f32(60, (5000,)),
    "sweep_outliers": lambda: synth.make_inputs("fp8_sweep_m65")[0],
    "exact_448": lambda: np.float32([448.0, -3.0, 1.0]),
    "just_above_448": lambda: np.float32([448.00003, 2.0]),
    "tiny": lambda: np.float32([1e-45, -3e-42, 1e-40]),
    "huge": lambda: np.float32([3.0e38, -1.0]),
    "zeros": lambda: np.zeros(100, np.float32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_pow2_scale_and_codes_bit_exact(name):
    x = CASES[name]()
    q, amax, scale = gpu_quantize_pow2(x)
    assert dg.dg_sync_status() == dg.DG_OK
    a_ref = oracle.amax(x)
    s_ref = oracle.scale_pow2_from_amax(a_ref)
    assert np.float32(scale[0].item()).view(np.uint32) == np.float32(s_ref).view(np.uint32), \
        (name, scale[0].item(), s_ref)
    assert np.array_equal(q.cpu().numpy().reshape(-1), oracle.quantize_e4m3(x, s_ref).reshape(-1))


def test_pow2_scale_special_values():
    for x in (np.float32([1.0, np.nan]), np.float32([np.inf, 1.0])):
        dx = dev(x)
        amax, scale = scalar(), scalar()
        dg.dg_amax_pow2(dx, amax, scale)
        assert dg.dg_sync_status() == dg.DG_OK
        s_ref = oracle.scale_pow2_from_amax(oracle.amax(x))
        got = scale[0].item()
        assert (np.isnan(got) and np.isnan(s_ref)) or got == s_ref


@pytest.mark.parametrize("M,N,K", [(1, 1000, 1040), (129, 1000, 1040), (640, 1536, 2048)])
def test_pow2_gemm_chain(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, _, sa = gpu_quantize_pow2(A)
    qb, _, sb = gpu_quantize_pow2(B)
    qa_ref, sa_ref, _ = oracle.quantize_tensor_pow2(A)
    qb_ref, sb_ref, _ = oracle.quantize_tensor_pow2(B)
    assert np.array_equal(qa.cpu().numpy(), qa_ref) and np.array_equal(qb.cpu().numpy(), qb_ref)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref)

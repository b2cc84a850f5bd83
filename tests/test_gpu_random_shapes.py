"""Seeded random shapes over every GEMM path the planner picks (warp-MMA GEMV,
CUDA-core GEMV layouts, split-K, single CTA, CTA pairs), E4M3 and FP16 inputs and each output type, every element checked
against the oracle and every byte around D checked untouched.  K is a
multiple of 16 (E4M3) or 8 (FP16), the only shape rule of the library."""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, check_guards, dev,
                     fp16_bits_to_f64, gpu_quantize, guarded, scalar)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def _shapes(seed, count):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        band = i % 4
        M = int(rng.integers(1, 17)) if band == 0 else int(rng.integers(17, 600)) if band < 3 \
            else int(rng.integers(256, 900))
        N = int(rng.integers(1, 1200))
        K = 16 * int(rng.integers(1, 130))
        out.append((M, N, K))
    return out


def _shapes_wide(seed, count):
    """Decode-style shapes: M <= 128 against wide B (N up to 13000), where
    the planner chooses between the warp-MMA GEMV, the CUDA-core GEMV,
    split-K (with its tile-aligned grid, staged fix-up and helper warps) and
    the tiled kernel."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        M = int(rng.integers(1, 3)) if i % 4 == 0 else int(rng.integers(3, 129))
        N = int(rng.integers(2000, 13000))
        K = 16 * int(rng.integers(16, 200))
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("M,N,K", _shapes(123, 24) + _shapes_wide(777, 16))
def test_random_fp8_shapes(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, _, sa_d = gpu_quantize(A)
    qb, _, sb_d = gpu_quantize(B)
    qa_ref, sa, _ = oracle.quantize_tensor(A)
    qb_ref, sb, _ = oracle.quantize_tensor(B)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    # BF16 output
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_fp8_gemm(qa, qb, D, sa_d, sb_d, None, dg.DG_BF16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb)
    # E4M3 output
    sd = np.float32(max(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))), 1e-30) / 448.0)
    sdt = scalar()
    sdt[0] = float(sd)
    buf8, D8 = guarded(M * N, torch.uint8, 0x7F)
    dg.dg_fp8_gemm(qa, qb, D8, sa_d, sb_d, sdt, dg.DG_E4M3, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf8, M * N, 0x7F)
    check_e4m3(D8.cpu().numpy().reshape(M, N), R, sa, sb, sd)


@pytest.mark.parametrize("M,N,K", [(m, n, k // 2) for (m, n, k) in _shapes(321, 12) + _shapes_wide(654, 6)])
def test_random_fp16_shapes(M, N, K):
    K = max(8, K - K % 8)
    A, B = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A.view(np.int16)), dev(B.view(np.int16)), D, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A, B)
    check_bf16_like(fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S,
                    1.0, 1.0, "FP16")

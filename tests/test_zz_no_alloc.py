"""dg_fp8_gemm_splitk_static (the split-K skinny GEMM on the library's fixed
static workspace, no allocation) against dg_fp8_gemm on the same split-K
path: two calls in a row, bit-identical results, error bits clear; one
shape also against the CPU oracle.  Self-contained, so it passes alone and
after the rest of the suite."""
import os

import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _parity import bf16_bits_to_f64, check_bf16_like, check_quantised, gpu_quantize, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def _inputs(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, amax_a, sa = gpu_quantize(A)
    qb, amax_b, sb = gpu_quantize(B)
    qa_ref, sa_ref = check_quantised(A, qa, amax_a, sa)
    qb_ref, sb_ref = check_quantised(B, qb, amax_b, sb)
    return qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref


@pytest.mark.parametrize("M,N,K,out", [
    (1, 1000, 1040, dg.DG_BF16),
    (3, 1000, 1040, dg.DG_BF16),
    (16, 12288, 512, dg.DG_BF16),    # tiles split over three CTAs
    (9, 2048, 2048, dg.DG_E4M3),
    (5, 300, 4096, dg.DG_FP16),
])
def test_static_workspace_matches_regular_entry(M, N, K, out):
    os.environ["DG_GEMV_MAX_M"] = "0"     # the regular entry takes the split-K path for M = 1 too
    dg.dg_reload_env()
    try:
        assert dg.dg_gemm_plan(M, N, K, dg.DG_E4M3, out)["path"] == 4
        qa, qb, sa, sb, *_ = _inputs(M, N, K)
        sd = scalar()
        sd[0] = 0.37
        dt = torch.uint8 if out == dg.DG_E4M3 else torch.int16
        ref = torch.empty((M, N), dtype=dt, device="cuda")
        dg.dg_fp8_gemm(qa, qb, ref, sa, sb, sd, out)
        assert dg.dg_sync_status() == dg.DG_OK
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
        for _ in range(2):            # two calls in a row on the same static workspace
            D = torch.full((M, N), 0x55, dtype=dt, device="cuda")
            dg.dg_fp8_gemm_splitk_static(qa, qb, D, sa, sb, sd, out, status_out=status)
            torch.cuda.synchronize()
            assert int(status[0].item()) == 0
            assert torch.equal(D, ref)
    finally:
        os.environ.pop("DG_GEMV_MAX_M", None)
        dg.dg_reload_env()


def test_static_workspace_matches_oracle():
    M, N, K = 12, 4000, 1024
    qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref = _inputs(M, N, K)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_splitk_static(qa, qb, D, sa, sb, None, dg.DG_BF16)
    torch.cuda.synchronize()
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref)

"""dg_fp8_gemm_splitk_static: the split-K skinny GEMM on the library's fixed
static workspace, for callers that cannot let a library allocate device
memory -- a process whose own pool allocator has reserved the device memory,
code that runs while a stream is captured in global mode (where cudaMalloc
is not allowed), or a latency-bound loop that cannot take cudaMalloc's
implicit synchronisation.

Checked here: against dg_fp8_gemm on the same split-K path (two calls in a
row, bit-identical, error bits clear); against the CPU oracle; a bounded
wait that runs out reported through status_out, then a correct call; free
device memory unchanged across calls, also in a fresh process whose first
library call is this one.  Self-contained, so it passes alone and after the
rest of the suite (this file is collected last)."""
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
    os.environ["DG_MMA_GEMV"] = "0"
    os.environ["DG_SPLITK"] = "1"         # and for 16 x 12288 x 512 (else the one-wave tiled kernel)
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
        os.environ.pop("DG_MMA_GEMV", None)
        os.environ.pop("DG_SPLITK", None)
        dg.dg_reload_env()


def test_static_workspace_matches_oracle():
    M, N, K = 12, 4000, 1024
    qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref = _inputs(M, N, K)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_splitk_static(qa, qb, D, sa, sb, None, dg.DG_BF16)
    torch.cuda.synchronize()
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref)


def test_static_workspace_timeout_sets_status_out_then_recovers():
    """A bounded wait that runs out on this entry point is reported through
    status_out (bit 1) and nowhere else; the next call, which zeroes the
    arrival counters again, is correct."""
    M, N, K = 8, 2048, 2048
    qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref = _inputs(M, N, K)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    assert dg.dg_sync_status() == dg.DG_OK
    dg.dg_set_wait_timeout_us(100_000)
    try:
        dg.dg_debug_skip_first_load(True)
        dg.dg_fp8_gemm_splitk_static(qa, qb, D, sa, sb, None, dg.DG_BF16, status_out=status)
        torch.cuda.synchronize()
        assert int(status[0].item()) & 1
    finally:
        dg.dg_set_wait_timeout_us(2_000_000)
        dg.dg_debug_skip_first_load(False)
    assert dg.dg_sync_status() == dg.DG_OK     # the library's own status word is untouched
    status.zero_()
    dg.dg_fp8_gemm_splitk_static(qa, qb, D, sa, sb, None, dg.DG_BF16, status_out=status)
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref)


def _calls_leave_free_memory_unchanged(qa, qb, D, sa, sb):
    dg.dg_fp8_gemm_splitk_static(qa, qb, D, sa, sb, None, dg.DG_BF16)   # warm-up (module load)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(4):
        dg.dg_fp8_gemm_splitk_static(qa, qb, D, sa, sb, None, dg.DG_BF16)
    torch.cuda.synchronize()
    return free0, torch.cuda.mem_get_info()[0]


def test_static_workspace_allocates_nothing():
    """Free device memory is the same before and after repeated calls."""
    M, N, K = 12, 4000, 1024
    qa, qb, sa, sb, *_ = _inputs(M, N, K)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    free0, free1 = _calls_leave_free_memory_unchanged(qa, qb, D, sa, sb)
    assert free1 == free0, (free0, free1)


def test_static_workspace_first_call_in_a_fresh_process():
    """In a new process whose first library call is this entry point (no
    dg_init, no other entry point): correct result, nothing allocated by
    the calls after the first."""
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = f"""
import sys
sys.path[:0] = [{os.path.dirname(here)!r}, {here!r}]
import numpy as np, torch
import fp16_tensor_core_gb300 as dg, oracle, synth
from _parity import bf16_bits_to_f64, check_bf16_like
from test_zz_no_alloc import _calls_leave_free_memory_unchanged
M, N, K = 9, 3000, 2048
A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
qa_ref, sa_ref, _ = oracle.quantize_tensor(A)
qb_ref, sb_ref, _ = oracle.quantize_tensor(B)
qa, qb = torch.from_numpy(qa_ref).cuda(), torch.from_numpy(qb_ref).cuda()
sa = torch.tensor([float(sa_ref)] * 4, device="cuda")
sb = torch.tensor([float(sb_ref)] * 4, device="cuda")
D = torch.empty((M, N), dtype=torch.int16, device="cuda")
free0, free1 = _calls_leave_free_memory_unchanged(qa, qb, D, sa, sb)
assert free1 == free0, (free0, free1)
R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref)
print("fresh ok")
"""
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "fresh ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])

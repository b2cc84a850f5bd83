"""Split-K tensor-core path for skinny GEMMs (plan path 4: M <= 16, and
M <= 128 where the tiled kernels would leave SMs idle; operands swapped, K blocks spread over every SM, partial tiles added in a fixed
order by the CTA that finishes a tile last) against the CPU oracle.

Covers ragged N (a partial last tile of 128 rows of B) and ragged K (a
zero-filled last K block), fewer K blocks than SMs, tiles split over two
and three CTAs, FP16 inputs, E4M3 output, run-to-run determinism, reuse of
the arrival counters across shapes and graph replays, and recovery after a
bounded wait runs out.  [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化
指南" §3.3 (M/N/K boundary handling)."""
import os

import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, check_guards,
                     check_quantised, dev, fp16_bits_to_f64, gpu_quantize, guarded,
                     sample_positions, scalar)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    # M <= 16 on this kernel, not the warp-MMA GEMV, and split-K for every
    # M <= 128 (over a short K with many tiles the default planner would take
    # the one-wave tiled kernel for some of these shapes)
    with knobs(DG_MMA_GEMV="0", DG_SPLITK="1"):
        yield
    assert dg.dg_sync_status() == dg.DG_OK


def _plan(M, N, K, in_dtype=dg.DG_E4M3):
    p = dg.dg_gemm_plan(M, N, K, in_dtype, dg.DG_BF16)
    assert p["path"] == 4, p
    return p


def _fp8_case(M, N, K, seed_name="fp8_sweep_m65"):
    A, B = synth.make_inputs(seed_name, M=M, N=N, K=K)
    qa, amax_a, sa = gpu_quantize(A)
    qb, amax_b, sb = gpu_quantize(B)
    qa_ref, sa_ref = check_quantised(A, qa, amax_a, sa)
    qb_ref, sb_ref = check_quantised(B, qb, amax_b, sb)
    return qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref


@pytest.mark.parametrize("M,N,K", [
    (3, 1000, 1040),     # ragged N and K; 8 tiles x 9 K blocks < 152 CTAs
    (16, 1000, 1040),
    (5, 128, 128),       # one tile, one K block
    (7, 300, 4096),      # 3 tiles x 32 K blocks over 96 CTAs
    (9, 2048, 2048),     # 16 x 16 = 256 units: tiles split over 2 CTAs
    (12, 4000, 1024),    # 32 x 8 = 256 units, ragged N
    (16, 12288, 512),    # 96 x 4 = 384 units: splits across 3 CTAs
    (4, 777, 16),        # K = 16: a single zero-filled K block
])
def test_splitk_bf16_matches_oracle(M, N, K):
    _plan(M, N, K)
    qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref = _fp8_case(M, N, K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    d = bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N))
    check_bf16_like(d, R, S, sa_ref, sb_ref)


@pytest.mark.parametrize("M,N,K", [
    (17, 1000, 1040),    # MMA N = 32
    (32, 4096, 1024),
    (33, 2000, 2048),    # MMA N = 64, ragged M
    (64, 4096, 4096),
    (65, 1000, 1040),    # MMA N = 128, ragged M; 8 tiles x 9 K blocks
    (100, 777, 3008),    # ragged N, 23.5 K blocks
    (128, 4096, 2048),
])
def test_splitk_wide_bf16_matches_oracle(M, N, K):
    """17 <= M <= 128: MMA N = 32 / 64 / 128 columns of A per CTA, the
    partial slots and the fixup walked 16 columns at a time."""
    p = _plan(M, N, K)
    assert p["block_m"] == (32 if M <= 32 else 64 if M <= 64 else 128), p
    qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref = _fp8_case(M, N, K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    d = bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N))
    check_bf16_like(d, R, S, sa_ref, sb_ref)


@pytest.mark.parametrize("M,N,K", [(48, 1000, 2080), (120, 640, 1040)])
def test_splitk_wide_e4m3_out_and_fp16(M, N, K):
    _plan(M, N, K)
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
    _plan(M, N, K, dg.DG_FP16)
    A16, B16 = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf16, D16 = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A16.view(np.int16)), dev(B16.view(np.int16)), D16, dg.DG_FP16,
                M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf16, M * N, 0x7FFF)
    R16, S16 = oracle.hgemm(A16, B16)
    check_bf16_like(fp16_bits_to_f64(D16.cpu().numpy().view(np.uint16).reshape(M, N)),
                    R16, S16, 1.0, 1.0, "FP16")


@pytest.mark.parametrize("M,N,K", [(48, 4096, 2048), (24, 2048, 1040)])
def test_splitk_staged_fixup_all_outputs(M, N, K):
    """Shapes whose finishing CTAs stage the other segments' partial tiles in
    shared memory (32 or 16 tiles, a whole multiple of CTAs per tile, every
    partial tile fits in the ring): BF16 and E4M3 out from E4M3 inputs and
    FP16 out from FP16 inputs."""
    p = _plan(M, N, K)
    assert p["grid"] % p["tiles"] == 0 and p["grid"] // p["tiles"] >= 2, p
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa_ref, sa, _ = oracle.quantize_tensor(A)
    qb_ref, sb, _ = oracle.quantize_tensor(B)
    qa, _, sa_d = gpu_quantize(A)
    qb, _, sb_d = gpu_quantize(B)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_fp8_gemm(qa, qb, D, sa_d, sb_d, None, dg.DG_BF16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb)
    sd = np.float32(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))) / 448.0)
    sdt = scalar()
    sdt[0] = float(sd)
    buf8, D8 = guarded(M * N, torch.uint8, 0x7F)
    dg.dg_fp8_gemm(qa, qb, D8, sa_d, sb_d, sdt, dg.DG_E4M3, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf8, M * N, 0x7F)
    check_e4m3(D8.cpu().numpy().reshape(M, N), R, sa, sb, sd)
    p16 = _plan(M, N, K, dg.DG_FP16)
    assert p16["grid"] % p16["tiles"] == 0, p16
    A16, B16 = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf16, D16 = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A16.view(np.int16)), dev(B16.view(np.int16)), D16, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf16, M * N, 0x7FFF)
    R16, S16 = oracle.hgemm(A16, B16)
    check_bf16_like(fp16_bits_to_f64(D16.cpu().numpy().view(np.uint16).reshape(M, N)), R16, S16,
                    1.0, 1.0, "FP16")


def test_splitk_m1_when_forced():
    """M = 1 and 2 on the split-K kernel (the GEMV crossover moved to 0)."""
    os.environ["DG_GEMV_MAX_M"] = "0"
    dg.dg_reload_env()
    try:
        for M in (1, 2):
            N, K = 1000, 1040
            _plan(M, N, K)
            qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref = _fp8_case(M, N, K)
            D = torch.empty((M, N), dtype=torch.int16, device="cuda")
            dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
            assert dg.dg_sync_status() == dg.DG_OK
            R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
            check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S,
                            sa_ref, sb_ref)
    finally:
        os.environ.pop("DG_GEMV_MAX_M", None)
        dg.dg_reload_env()


def test_splitk_qkv_m16_all_outputs():
    """The decode QKV weight shape with 16 activation rows, every output."""
    M, N, K = 16, 12288, 4096
    _plan(M, N, K)
    A, B = synth.make_inputs("fp8_qkv", M=M)
    qa, amax_a, sa = gpu_quantize(A)
    qb, amax_b, sb = gpu_quantize(B)
    qa_ref, sa_ref = check_quantised(A, qa, amax_a, sa)
    qb_ref, sb_ref = check_quantised(B, qb, amax_b, sb)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    d = bf16_bits_to_f64(D.cpu().numpy().view(np.uint16))
    check_bf16_like(d, R, S, sa_ref, sb_ref)


def test_splitk_e4m3_out():
    M, N, K = 11, 1000, 2080
    _plan(M, N, K)
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


@pytest.mark.parametrize("M,N,K", [(3, 520, 1040), (16, 1000, 3000)])
def test_splitk_fp16_hgemm(M, N, K):
    _plan(M, N, K, dg.DG_FP16)
    A, B = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A.view(np.int16)), dev(B.view(np.int16)), D, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A, B)
    check_bf16_like(fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S,
                    1.0, 1.0, "FP16")


def test_splitk_deterministic_and_counters_reused_across_shapes():
    """Partial tiles are added in segment order, so repeated calls give the
    same bits; interleaving shapes with different tile splits reuses the
    arrival counters, which every call must leave at zero."""
    shapes = [(9, 2048, 2048), (16, 12288, 512), (3, 1000, 1040)]
    cases = [(s, _fp8_case(*s)) for s in shapes]
    first = {}
    for rep in range(3):
        for (M, N, K), (qa, qb, sa, sb, *_rest) in cases:
            D = torch.empty((M, N), dtype=torch.int16, device="cuda")
            dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
            assert dg.dg_sync_status() == dg.DG_OK
            h = D.cpu().numpy()
            if rep == 0:
                first[(M, N, K)] = h
            else:
                assert np.array_equal(h, first[(M, N, K)]), (M, N, K, rep)
    M, N, K = shapes[1]
    _, _, _, _, qa_ref, qb_ref, sa_ref, sb_ref = cases[1][1]
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(first[(M, N, K)].view(np.uint16)), R, S, sa_ref, sb_ref)


def test_splitk_graph_replay():
    M, N, K = 16, 12288, 512
    qa, qb, sa, sb, *_ = _fp8_case(M, N, K)
    direct = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm(qa, qb, direct, sa, sb, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    D = torch.empty_like(direct)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):   # three launches per replay: counters must be back at zero each time
            dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, stream=s)
    for _ in range(2):
        D.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert dg.dg_sync_status() == dg.DG_OK
        assert torch.equal(D, direct)


@pytest.mark.parametrize("M,N,K", [(64, 4096, 4096), (16, 1024, 4096), (24, 2048, 1040)])
def test_splitk_staged_fixup_repeatable_back_to_back(M, N, K):
    """Eight launches per graph replay, 50 replays: every output equals the
    first launch's bit for bit.  The finishing CTAs copy the other segments'
    partial tiles into shared memory with bulk copies after their acquiring
    arrival atomic; a missing ordering would show as an occasional stale
    partial, so a different sum."""
    p = _plan(M, N, K)
    assert p["grid"] % p["tiles"] == 0
    qa, qb, sa, sb, *_ = _fp8_case(M, N, K)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm(qa, qb, ref, sa, sb, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    outs = [torch.empty_like(ref) for _ in range(8)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for D in outs:
            dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for D in outs:
            dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, stream=s)
    for r in range(50):
        g.replay()
        if r % 10 == 9:
            torch.cuda.synchronize()
            for D in outs:
                assert torch.equal(D, ref)
    torch.cuda.synchronize()
    assert dg.dg_sync_status() == dg.DG_OK


def test_splitk_timeout_then_recovers():
    """One stage left unloaded: the bounded wait runs out, the call reports
    DG_ERR_TIMEOUT, dg_sync_status clears the arrival counters, and the next
    split-K GEMM is correct."""
    M, N, K = 9, 2048, 2048
    _plan(M, N, K)
    qa, qb, sa, sb, qa_ref, qb_ref, sa_ref, sb_ref = _fp8_case(M, N, K)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    assert dg.dg_sync_status() == dg.DG_OK
    dg.dg_set_wait_timeout_us(100_000)
    try:
        dg.dg_debug_skip_first_load(True)
        dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
        assert dg.dg_sync_status() == dg.DG_ERR_TIMEOUT
        assert dg.dg_sync_status() == dg.DG_OK
    finally:
        dg.dg_set_wait_timeout_us(2_000_000)
        dg.dg_debug_skip_first_load(False)
    D.zero_()
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa_ref, sb_ref)


def test_splitk_two_streams_concurrently():
    """Split-K GEMMs issued on two streams without ordering between them give
    the same bits as on one stream: each stream has its own workspace."""
    shapes = [(9, 2048, 2048), (16, 12288, 512)]
    cases = [_fp8_case(*sh) for sh in shapes]
    ref = []
    for (M, N, K), (qa, qb, sa, sb, *_r) in zip(shapes, cases):
        D = torch.empty((M, N), dtype=torch.int16, device="cuda")
        dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16)
        ref.append(D)
    assert dg.dg_sync_status() == dg.DG_OK
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[torch.empty_like(r) for _ in range(6)] for r in ref]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for i in range(6):
        for j, ((qa, qb, sa, sb, *_r), st) in enumerate(zip(cases, streams)):
            dg.dg_fp8_gemm(qa, qb, outs[j][i], sa, sb, None, dg.DG_BF16, stream=st)
    torch.cuda.synchronize()
    assert dg.dg_sync_status() == dg.DG_OK
    for j in range(2):
        for o in outs[j]:
            assert torch.equal(o, ref[j])

"""Split-K row ranges (DG_SPLITK_ROWS=1: plan path 4 with block_n < 128)
against the oracle.

With N within 128 rows per SM, each CTA owns ceil(N / SMs) rows of B over
the whole of K: no tile is split, so no partial tile, workspace or finishing
pass.  The TMA box is the row range; the MMA still spans 128 rows and the
rows past the range are never stored.  Every output is compared; guard
regions around D catch stores outside [0, M) x [0, N), in particular rows of
one range written by the CTA of the range before it.  Shapes: the decode QKV
and FFN-down projections, ragged ranges (7 rows), one row per CTA, K tails
and K shorter than one K block, FP16 operands, E4M3 output, the output-amax
report, M > 16 when forced, repeatability, and a graph capture on a stream
that never ran a split-K GEMM (no workspace to allocate).
"""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, check_guards, dev,
                     fp16_bits_to_f64, gpu_quantize, guarded, scalar)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    # M <= 8 on split-K instead of the warp-MMA GEMV; row ranges
    # split-K for every M <= 128: over a short K with many tiles the default
    # planner takes the one-wave tiled kernel for some of these shapes
    with knobs(DG_MMA_GEMV="0", DG_SPLITK="1", DG_SPLITK_ROWS="1"):
        yield
    assert dg.dg_sync_status() == dg.DG_OK


def _plan(M, N, K, in_dtype=dg.DG_E4M3, out=dg.DG_BF16):
    p = dg.dg_gemm_plan(M, N, K, in_dtype, out)
    assert p["path"] == 4 and p["block_n"] < 128 and p["grid"] == p["tiles"], p
    return p


def _quantised(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa_ref, sa, _ = oracle.quantize_tensor(A)
    qb_ref, sb, _ = oracle.quantize_tensor(B)
    return qa_ref, qb_ref, sa, sb


def _scales(sa, sb):
    sat, sbt = scalar(), scalar()
    sat[0], sbt[0] = float(sa), float(sb)
    return sat, sbt


@pytest.mark.parametrize("M,N,K", [
    (16, 12288, 4096),   # decode QKV: 81 rows per CTA
    (9, 4096, 11008),    # decode FFN down: 27 rows per CTA, long K
    (3, 1000, 1040),     # 7 rows per CTA, ragged last range, K tail
    (16, 17, 16),        # one row per CTA, K shorter than one K block
    (7, 5000, 272),      # 33 rows, K tail
    (12, 300, 4096),     # 2 rows per CTA
])
def test_bf16_out(M, N, K):
    _plan(M, N, K)
    qa_ref, qb_ref, sa, sb = _quantised(M, N, K)
    sat, sbt = _scales(sa, sb)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    am = scalar()
    dg.dg_fp8_gemm_amax(dev(qa_ref), dev(qb_ref), D, sat, sbt, None, dg.DG_BF16, am,
                        M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb)
    ref = float(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))))
    i = np.argmax(np.abs(R))
    tol = 8e-3 * ref + 1e-4 * S.reshape(-1)[i] * float(sa) * float(sb)
    assert abs(am[0].item() - ref) <= tol, (am[0].item(), ref, tol)


@pytest.mark.parametrize("M,N,K", [(16, 12288, 1024), (5, 999, 528)])
def test_e4m3_out(M, N, K):
    qa_ref, qb_ref, sa, sb = _quantised(M, N, K)
    sat, sbt = _scales(sa, sb)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    # a median-based output scale: many codes saturate at +-448
    sd = np.float32(np.median(np.abs(oracle.epilogue_scale(R, sa, sb))) / 64.0)
    sdt = scalar()
    sdt[0] = float(sd)
    buf, D = guarded(M * N, torch.uint8, 0x7F)
    _plan(M, N, K, out=dg.DG_E4M3)
    dg.dg_fp8_gemm(dev(qa_ref), dev(qb_ref), D, sat, sbt, sdt, dg.DG_E4M3, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F)
    check_e4m3(D.cpu().numpy().reshape(M, N), R, sa, sb, sd)


@pytest.mark.parametrize("M,N,K", [(16, 12288, 4096), (4, 1000, 1040), (13, 4096, 272)])
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


@pytest.mark.parametrize("M,N,K", [(64, 4096, 4096), (128, 2000, 1040), (33, 12288, 512)])
def test_wide_a_when_forced(M, N, K):
    with knobs(DG_SPLITK="1", DG_SPLITK_ROWS="1"):
        p = _plan(M, N, K)
        assert p["block_m"] == (64 if M <= 64 else 128), p
        qa_ref, qb_ref, sa, sb = _quantised(M, N, K)
        sat, sbt = _scales(sa, sb)
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
        dg.dg_fp8_gemm(dev(qa_ref), dev(qb_ref), D, sat, sbt, None, dg.DG_BF16, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb)


def test_repeatable_and_graph_capture_on_a_fresh_stream():
    M, N, K = 16, 12288, 2048
    _plan(M, N, K)
    qa_ref, qb_ref, sa, sb = _quantised(M, N, K)
    sat, sbt = _scales(sa, sb)
    qa, qb = dev(qa_ref), dev(qb_ref)
    D0 = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm(qa, qb, D0, sat, sbt, None, dg.DG_BF16)
    outs = [torch.empty_like(D0) for _ in range(4)]
    for o in outs:
        dg.dg_fp8_gemm(qa, qb, o, sat, sbt, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    for o in outs:
        assert torch.equal(o, D0)   # one CTA per range, fixed order: the same bits
    # a stream that never ran a split-K GEMM can be captured: nothing to allocate
    s = torch.cuda.Stream()
    Dg = torch.zeros_like(D0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dg.dg_fp8_gemm(qa, qb, Dg, sat, sbt, None, dg.DG_BF16, stream=s.cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    assert dg.dg_sync_status() == dg.DG_OK
    assert torch.equal(Dg, D0)


@pytest.mark.parametrize("rows", ["64", "32"])
@pytest.mark.parametrize("M,N,K", [(16, 12288, 4096), (5, 1000, 1040), (12, 4096, 11008)])
def test_short_split_tiles(rows, M, N, K):
    """Split-K over tiles shorter than 128 rows (DG_SPLITK_TILE_ROWS): tiles
    split between CTAs whose accumulators hold rows past the tile (stale
    shared memory), which the finishing pass adds but never stores."""
    with knobs(DG_SPLITK_ROWS="0", DG_SPLITK_TILE_ROWS=rows):
        p = dg.dg_gemm_plan(M, N, K)
        assert p["path"] == 4 and p["block_n"] == int(rows) and p["grid"] != p["tiles"], p
        qa_ref, qb_ref, sa, sb = _quantised(M, N, K)
        sat, sbt = _scales(sa, sb)
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
        am = scalar()
        dg.dg_fp8_gemm_amax(dev(qa_ref), dev(qb_ref), D, sat, sbt, None, dg.DG_BF16, am,
                            M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb)
    ref = float(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))))
    i = np.argmax(np.abs(R))
    tol = 8e-3 * ref + 1e-4 * S.reshape(-1)[i] * float(sa) * float(sb)
    assert abs(am[0].item() - ref) <= tol, (am[0].item(), ref, tol)

"""CTA-pair GEMM with a split tail (DG_SPLIT_TAIL=1; measured no faster than
whole tiles on GB300, so off by default): when the tiles do not fill the
last wave of pairs, the kernel cuts each remaining tile into 2-4 K ranges
over the otherwise idle pairs; the pair holding the first range adds the
others' FP32 partial tiles in range order and stores the tile.  Checked against
the oracle on every output ([FP8-guide] §3.1's K-blocked accumulation, §3.3
edges), for 2, 3 and 4 ranges per tile (which of them a shape gets depends
on how many pairs the GPU runs at once, so several shapes are used), ragged
M / N / K, E4M3 and FP16 outputs, FP16 operands, the output-amax report,
and bit-for-bit repeatability (the ranges are added in a fixed order)."""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, check_guards, dev,
                     fp16_bits_to_f64, guarded, scalar)

pytestmark = pytest.mark.gpu

# 256 x 256 pair tiles (forced), so that the tile count is known: with 76
# pairs, 95 tiles leave 19 (4 ranges each), 100 leave 24 (3), 108 leave 32
# (2); other pair counts land on other splits.
SHAPES = [
    (1280, 4864, 1024),   # 5 x 19 = 95 tiles
    (1200, 5000, 1040),   # 5 x 20 = 100 tiles, ragged M, N and K
    (1536, 4608, 2048),   # 6 x 18 = 108 tiles
    (2304, 4352, 512),    # 9 x 17 = 153 tiles: two full waves and one tile
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    with knobs(DG_2CTA="1", DG_FORCE_BLOCK_N="256", DG_SPLIT_TAIL="1"):
        yield
    assert dg.dg_sync_status() == dg.DG_OK


def _codes(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, sa, _ = oracle.quantize_tensor(A)
    qb, sb, _ = oracle.quantize_tensor(B)
    sat, sbt = scalar(), scalar()
    sat[0], sbt[0] = float(sa), float(sb)
    return qa, qb, sa, sb, sat, sbt


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_split_tail_bf16_matches_oracle(M, N, K):
    p = dg.dg_gemm_plan(M, N, K)
    assert (p["block_m"], p["block_n"]) == (256, 256), p
    qa, qb, sa, sb, sat, sbt = _codes(M, N, K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_fp8_gemm(dev(qa), dev(qb), D, sat, sbt, None, dg.DG_BF16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa, qb)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb)


@pytest.mark.parametrize("M,N,K", SHAPES[:2])
def test_split_tail_e4m3_fp16_out_and_amax(M, N, K):
    qa, qb, sa, sb, sat, sbt = _codes(M, N, K)
    R, S = oracle.gemm_e4m3(qa, qb)
    dref = oracle.epilogue_scale(R, sa, sb)
    sd = np.float32(np.median(np.abs(dref)) / 64.0)
    sdt = scalar()
    sdt[0] = float(sd)
    buf, D = guarded(M * N, torch.uint8, 0x7F)
    am = scalar()
    dg.dg_fp8_gemm_amax(dev(qa), dev(qb), D, sat, sbt, sdt, dg.DG_E4M3, am, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F)
    check_e4m3(D.cpu().numpy().reshape(M, N), R, sa, sb, sd)
    i = np.argmax(np.abs(dref))
    ref = float(np.abs(dref.reshape(-1)[i]))
    tol = 8e-3 * ref + 1e-4 * float(S.reshape(-1)[i]) * float(sa) * float(sb)
    assert abs(am[0].item() - ref) <= tol, (am[0].item(), ref, tol)
    buf16, D16 = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_fp8_gemm(dev(qa), dev(qb), D16, sat, sbt, None, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf16, M * N, 0x7FFF)
    check_bf16_like(fp16_bits_to_f64(D16.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb,
                    "FP16")


@pytest.mark.parametrize("M,N,K", [(1280, 4864, 1024), (1200, 5000, 1040)])
def test_split_tail_fp16_operands(M, N, K):
    A16, B16 = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A16.view(np.int16)), dev(B16.view(np.int16)), D, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A16, B16)
    check_bf16_like(fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, 1.0, 1.0,
                    "FP16")


def test_split_tail_repeatable_and_close_to_unsplit():
    """Back-to-back launches give the same bits (fixed range order), and the
    result is within the tolerance of the same GEMM without the split."""
    M, N, K = 1280, 4864, 1024
    qa, qb, sa, sb, sat, sbt = _codes(M, N, K)
    dqa, dqb = dev(qa), dev(qb)
    outs = [torch.empty((M, N), dtype=torch.int16, device="cuda") for _ in range(6)]
    for o in outs:
        dg.dg_fp8_gemm(dqa, dqb, o, sat, sbt, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    with knobs(DG_SPLIT_TAIL="0"):
        whole = torch.empty_like(outs[0])
        dg.dg_fp8_gemm(dqa, dqb, whole, sat, sbt, None, dg.DG_BF16)
        assert dg.dg_sync_status() == dg.DG_OK
    R, S = oracle.gemm_e4m3(qa, qb)
    for D in (outs[0], whole):
        check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa, sb)


def test_split_tail_timeout_then_recovers():
    """A stage left unloaded in the first CTA: its bounded waits run out, the
    tile's finishing CTA may give up waiting for a missing range; the call
    reports DG_ERR_TIMEOUT, dg_sync_status clears the arrival counters, and
    the next call is correct."""
    M, N, K = 1280, 4864, 1024
    qa, qb, sa, sb, sat, sbt = _codes(M, N, K)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    assert dg.dg_sync_status() == dg.DG_OK
    dg.dg_set_wait_timeout_us(100_000)
    try:
        dg.dg_debug_skip_first_load(True)
        dg.dg_fp8_gemm(dev(qa), dev(qb), D, sat, sbt, None, dg.DG_BF16)
        assert dg.dg_sync_status() == dg.DG_ERR_TIMEOUT
        assert dg.dg_sync_status() == dg.DG_OK
    finally:
        dg.dg_set_wait_timeout_us(2_000_000)
        dg.dg_debug_skip_first_load(False)
    dg.dg_fp8_gemm(dev(qa), dev(qb), D, sat, sbt, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    R, S = oracle.gemm_e4m3(qa, qb)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S, sa, sb)

"""The CTA-pair GEMM under the stream-K schedule (DG_STREAM_K=1) against the
oracle.

The (tile, K block) units of all tiles are cut into one equal range per pair;
a tile cut at a boundary is split in two, the later K range published as an
FP32 partial tile by the pair that starts with it, the first K range run last
by the pair before, which adds the partial and stores the tile.  Each case
checks from the DG_LOG line that the schedule ran, and compares every
output: ragged M and N with a K tail, a K of a few blocks, E4M3 and FP16
outputs, FP16 operands, the output-amax report and repeatability (the two
halves of a split tile are added in a fixed order).
"""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    with knobs(DG_2CTA="1", DG_FORCE_BLOCK_N="256", DG_STREAM_K="1", DG_LOG="1"):
        yield
    assert dg.dg_sync_status() == dg.DG_OK


def _ran_stream_k(capfd):
    err = capfd.readouterr().err
    assert "stream-K" in err, err[-2000:]


def _quantised(M, N, K):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa_ref, sa, _ = oracle.quantize_tensor(A)
    qb_ref, sb, _ = oracle.quantize_tensor(B)
    sat, sbt = scalar(), scalar()
    sat[0], sbt[0] = float(sa), float(sb)
    return qa_ref, qb_ref, sa, sb, sat, sbt


@pytest.mark.parametrize("M,N,K", [
    (4800, 2250, 1040),   # 19 x 9 = 171 tiles over 76 pairs, ragged M, N and K
    (4096, 4096, 512),    # 256 tiles of 4 K blocks
])
def test_bf16_out_and_amax(M, N, K, capfd):
    qa_ref, qb_ref, sa, sb, sat, sbt = _quantised(M, N, K)
    p = dg.dg_gemm_plan(M, N, K)
    assert p["path"] == 3 and p["block_m"] == 256 and p["block_n"] == 256, p
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    am = scalar()
    dg.dg_fp8_gemm_amax(dev(qa_ref), dev(qb_ref), D, sat, sbt, None, dg.DG_BF16, am, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    _ran_stream_k(capfd)
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, sa, sb)
    ref = float(np.max(np.abs(oracle.epilogue_scale(R, sa, sb))))
    i = np.argmax(np.abs(R))
    tol = 8e-3 * ref + 1e-4 * S.reshape(-1)[i] * float(sa) * float(sb)
    assert abs(am[0].item() - ref) <= tol, (am[0].item(), ref, tol)


def test_e4m3_out(capfd):
    M, N, K = 4800, 2304, 1040
    qa_ref, qb_ref, sa, sb, sat, sbt = _quantised(M, N, K)
    R = oracle.gemm_e4m3(qa_ref, qb_ref, with_abs=False)
    sd = np.float32(np.median(np.abs(oracle.epilogue_scale(R, sa, sb))) / 64.0)
    sdt = scalar()
    sdt[0] = float(sd)
    buf, D = guarded(M * N, torch.uint8, 0x7F)
    dg.dg_fp8_gemm(dev(qa_ref), dev(qb_ref), D, sat, sbt, sdt, dg.DG_E4M3, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    _ran_stream_k(capfd)
    check_guards(buf, M * N, 0x7F)
    check_e4m3(D.cpu().numpy().reshape(M, N), R, sa, sb, sd)


def test_fp16_operands(capfd):
    M, N, K = 4608, 2200, 1000
    A16, B16 = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    dg.dg_hgemm(dev(A16.view(np.int16)), dev(B16.view(np.int16)), D, dg.DG_FP16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    _ran_stream_k(capfd)
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A16, B16)
    check_bf16_like(fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, 1.0, 1.0,
                    "FP16")


def test_repeatable(capfd):
    M, N, K = 4096, 4608, 768
    qa_ref, qb_ref, _, _, sat, sbt = _quantised(M, N, K)
    qa, qb = dev(qa_ref), dev(qb_ref)
    outs = [torch.empty((M, N), dtype=torch.int16, device="cuda") for _ in range(5)]
    for o in outs:
        dg.dg_fp8_gemm(qa, qb, o, sat, sbt, None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    _ran_stream_k(capfd)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])

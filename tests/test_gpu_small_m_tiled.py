"""The single-CTA tiled kernel for short operands and ragged edges, with
each box height (full: 128 rows of A, BN of B; the operand's rows rounded
up to 8 when it has at most 32; the last tile's rows rounded up to 8
whenever an operand ends inside a tile, the default), against the oracle.

The MMA always reads 128 rows of A and BN of B from shared memory; with a
shorter box the rows past it hold whatever the stage held before, and only
output rows past M or columns past N depend on them, which are neither
stored nor counted in the output amax.  Shapes: M = 1..100 forced onto the
tiled path (GEMV, warp-MMA GEMV and split-K off), N = 8..32 (the 64-wide
tile over a short B), both short, M = 129 and 300 (an edge tile of 1 and
44 rows) with ragged N, and a K tail, E4M3 and FP16
operands, BF16 and E4M3 output with the amax report; guard sentinels
around D.
"""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import (bf16_bits_to_f64, check_bf16_like, check_e4m3, check_guards, dev,
                     gpu_quantize, guarded, scalar)

pytestmark = pytest.mark.gpu

TILED = dict(DG_GEMV_MAX_M="0", DG_MMA_GEMV="0", DG_SPLITK="0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


@pytest.mark.parametrize("box", ["0", "1", "2"])
@pytest.mark.parametrize("M,N", [(1, 1000), (8, 1000), (17, 1000), (31, 1000), (32, 1000),
                                 (33, 1000), (100, 1000), (300, 8), (300, 17), (700, 31),
                                 (300, 32), (17, 9), (129, 1000), (300, 777)])
@pytest.mark.parametrize("out", [dg.DG_BF16, dg.DG_E4M3])
def test_e4m3_small_m(box, M, N, out):
    K = 1040
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, _, sa = gpu_quantize(A)
    qb, _, sb = gpu_quantize(B)
    qa_ref, sa_ref, _ = oracle.quantize_tensor(A)
    qb_ref, sb_ref, _ = oracle.quantize_tensor(B)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    sd_val, sd = None, None
    if out == dg.DG_E4M3:
        sd_val = np.float32(np.max(np.abs(oracle.epilogue_scale(R, sa_ref, sb_ref))) / 448.0)
        sd = scalar()
        sd[0] = float(sd_val)
        buf, D = guarded(M * N, torch.uint8, 0x7F)
    else:
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
    am = scalar()
    with knobs(DG_TC_SHORT_BOX=box, **TILED):
        plan = dg.dg_gemm_plan(M, N, K, dg.DG_E4M3, out)
        assert (plan["path"], plan["block_m"]) == (3, 128), plan
        dg.dg_fp8_gemm_amax(qa, qb, D, sa, sb, sd, out, am, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F if out == dg.DG_E4M3 else 0x7FFF)
    h = D.cpu().numpy()
    if out == dg.DG_E4M3:
        check_e4m3(h.reshape(M, N), R, sa_ref, sb_ref, sd_val)
    else:
        check_bf16_like(bf16_bits_to_f64(h.view(np.uint16).reshape(M, N)), R, S, sa_ref, sb_ref)
    ref_am = float(np.max(np.abs(oracle.epilogue_scale(R, sa_ref, sb_ref))))
    i = np.argmax(np.abs(R))
    tol = 8e-3 * ref_am + 1e-4 * S.reshape(-1)[i] * float(sa_ref) * float(sb_ref)
    assert abs(am[0].item() - ref_am) <= tol, (am[0].item(), ref_am, tol)


@pytest.mark.parametrize("box", ["0", "1", "2"])
@pytest.mark.parametrize("M,N", [(3, 777), (24, 777), (57, 777), (500, 24)])
def test_fp16_small_m(box, M, N):
    K = 1000
    A, B = synth.make_inputs("fp16_4096", M=M, N=N, K=K)
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    with knobs(DG_TC_SHORT_BOX=box, **TILED):
        plan = dg.dg_gemm_plan(M, N, K, dg.DG_FP16, dg.DG_BF16)
        assert (plan["path"], plan["block_m"]) == (3, 128), plan
        dg.dg_hgemm(dev(A.view(np.int16)), dev(B.view(np.int16)), D, dg.DG_BF16, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A, B)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S, 1.0, 1.0)

"""The tiled kernels' staged epilogue at tile widths with an odd number of
32-column chunks, against the oracle.

Each CTA's last tile gives every 32 x 32 output box its own place in the
drained operand ring and stores them together; earlier tiles go through one
staging box per warp.  Shapes cover whole and ragged last tiles, several
tiles per CTA, widths of 224, 160 and 96 columns (7, 5 and 3 chunks), rows past M
in the odd CTA of a pair, both kernels, BF16 and E4M3 output (E4M3 rows of
1000 bytes are not 16-byte multiples and take the direct stores), the
output-amax report and the grouped kernel.  Every element is compared.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


@pytest.mark.parametrize("kernel,bn", [("1", None), ("0", None), ("1", "224"), ("1", "160"),
                                       ("0", "224"), ("0", "160"), ("0", "96")])
@pytest.mark.parametrize("M,N,K", [
    (300, 1000, 272),    # ragged N, odd CTA's rows past M, one tile per CTA
    (640, 2240, 1040),   # several tiles per CTA, K tail
])
@pytest.mark.parametrize("out", [dg.DG_BF16, dg.DG_E4M3])
def test_odd_chunk_widths(kernel, bn, M, N, K, out):
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, _, sa = gpu_quantize(A)
    qb, _, sb = gpu_quantize(B)
    qa_ref, sa_ref, _ = oracle.quantize_tensor(A)
    qb_ref, sb_ref, _ = oracle.quantize_tensor(B)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    sd_val, sd = None, None
    if out == dg.DG_E4M3:
        # a median-based output scale: many codes saturate, exercising the clamp
        sd_val = np.float32(np.median(np.abs(oracle.epilogue_scale(R, sa_ref, sb_ref))) / 64.0)
        sd = scalar()
        sd[0] = float(sd_val)
        buf, D = guarded(M * N, torch.uint8, 0x7F)
    else:
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
    am = scalar()
    with knobs(DG_2CTA=kernel, DG_FORCE_BLOCK_N=bn):
        plan = dg.dg_gemm_plan(M, N, K, dg.DG_E4M3, out)
        assert plan["path"] == 3 and plan["block_m"] == (256 if kernel == "1" else 128), plan
        if bn is not None:
            assert plan["block_n"] == int(bn), plan
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


@pytest.mark.parametrize("N", [400, 1000])   # 128- and 256-wide tiles, ragged last column
def test_grouped_widths(N):
    G, total, K = 6, 2000, 1024
    A, B, offs = synth.make_moe_inputs(G, total, N, K, seed=3, empty=1)
    # the codes of every slice are exact E4M3 values at scale 1
    qa = dev(oracle.e4m3_encode(A.astype(np.float64)))
    qb = dev(oracle.e4m3_encode(B.astype(np.float64)))
    sa = torch.ones(G, dtype=torch.float32, device="cuda")
    sb = torch.full((G,), 0.5, dtype=torch.float32, device="cuda")
    D = torch.full((total, N), 0x7FFF, dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_grouped(qa, qb, D, dev(offs), sa, sb, None, dg.DG_BF16, M=total, N=N, K=K,
                           groups=G)
    assert dg.dg_sync_status() == dg.DG_OK
    h = D.cpu().numpy().view(np.uint16)
    qa_h, qb_h = qa.cpu().numpy(), qb.cpu().numpy()
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        if r1 == r0:
            continue
        R, S = oracle.gemm_e4m3(qa_h[r0:r1], qb_h[g * N:(g + 1) * N])
        check_bf16_like(bf16_bits_to_f64(h[r0:r1]), R, S, 1.0, 0.5, f"group {g}")


@pytest.mark.parametrize("M,N,K,fp16", [
    (48, 11008, 1040, False),   # 115 tiles of 128 x 96, the last 64 wide; K tail
    (32, 12288, 4096, False),   # the decode QKV projection at a batch of 32
    (17, 14336, 1040, True),    # FP16 operands
    (16, 12288, 1040, False),   # 16 rows over a short K: tiled instead of split-K
    (12, 11008, 2048, False),   # two K blocks per stage
    (40, 12288, 1664, False),   # 13 K blocks, two per stage: the last stage's second is past K
])
def test_one_wave_96_wide(M, N, K, fp16):
    """Shapes whose every tile fits one wave only at 96 columns take the
    96-wide single-CTA tile from the default planner (at 9..16 rows only over
    a short K); every element against the oracle."""
    plan = dg.dg_gemm_plan(M, N, K, dg.DG_FP16 if fp16 else dg.DG_E4M3, dg.DG_BF16)
    assert (plan["path"], plan["block_m"], plan["block_n"]) == (3, 128, 96), plan
    assert plan["tiles"] == (N + 95) // 96 <= plan["grid"], plan
    buf, D = guarded(M * N, torch.int16, 0x7FFF)
    if fp16:
        ha, hb = synth.make_inputs("fp16_4096", M=M, N=N, K=K)   # binary16 bit patterns
        dg.dg_hgemm(dev(ha.view(np.int16)), dev(hb.view(np.int16)), D, dg.DG_BF16, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
        R, S = oracle.hgemm(ha, hb)
        check_guards(buf, M * N, 0x7FFF)
        check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S,
                        1.0, 1.0)
        return
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, _, sa = gpu_quantize(A)
    qb, _, sb = gpu_quantize(B)
    qa_ref, sa_ref, _ = oracle.quantize_tensor(A)
    qb_ref, sb_ref, _ = oracle.quantize_tensor(B)
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, None, dg.DG_BF16, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    check_guards(buf, M * N, 0x7FFF)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N)), R, S,
                    sa_ref, sb_ref)

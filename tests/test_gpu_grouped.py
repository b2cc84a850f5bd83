"""Grouped E4M3 GEMM (dg_fp8_gemm_grouped) against the oracle, group by group,
and against one dg_fp8_gemm call per group.  Group sizes come from the skewed
MoE recipe in `synth` (empty groups, sizes that straddle 128-row tiles)."""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _parity import bf16_bits_to_f64, check_bf16_like, check_e4m3, dev, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def quantise_groups(A, B, offs, N):
    """Per-group per-tensor quantisation on the GPU (one dg_amax + quantise
    per slice) and in the oracle; returns device codes and scales and the
    oracle's codes and scales."""
    G = len(offs) - 1
    qa = torch.empty(A.shape, dtype=torch.uint8, device="cuda")
    qb = torch.empty(B.shape, dtype=torch.uint8, device="cuda")
    sa = torch.ones(G, dtype=torch.float32, device="cuda")
    sb = torch.ones(G, dtype=torch.float32, device="cuda")
    dA, dB = dev(A), dev(B)
    ref = []
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        am = scalar()
        bsl = slice(g * N, (g + 1) * N)
        dg.dg_amax(dB[bsl], am, sb[g:g + 1])
        dg.dg_quantize_e4m3(dB[bsl], sb[g:g + 1], qb[bsl])
        qb_r, sb_r, _ = oracle.quantize_tensor(B[bsl])
        if r1 > r0:
            dg.dg_amax(dA[r0:r1], am, sa[g:g + 1])
            dg.dg_quantize_e4m3(dA[r0:r1], sa[g:g + 1], qa[r0:r1])
            qa_r, sa_r, _ = oracle.quantize_tensor(A[r0:r1])
        else:
            qa_r, sa_r = np.zeros((0, A.shape[1]), np.uint8), np.float32(1.0)
        ref.append((qa_r, sa_r, qb_r, sb_r))
    assert dg.dg_sync_status() == dg.DG_OK
    return qa, qb, sa, sb, ref


@pytest.mark.parametrize("G,total,N,K,empty", [
    (8, 1500, 1000, 1040, 1),    # ragged sizes, one empty group, N not a tile multiple
    (16, 4096, 512, 512, 2),     # many groups
    (3, 300, 256, 256, 0),       # small
    (1, 777, 640, 272, 0),       # a single group
])
def test_grouped_bf16_matches_oracle(G, total, N, K, empty):
    A, B, offs = synth.make_moe_inputs(G, total, N, K, empty=empty)
    qa, qb, sa, sb, ref = quantise_groups(A, B, offs, N)
    D = torch.full((total, N), 0x7FFF, dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_grouped(qa, qb, D, dev(offs), sa, sb, None, dg.DG_BF16, M=total, N=N, K=K,
                           groups=G)
    assert dg.dg_sync_status() == dg.DG_OK
    h = D.cpu().numpy().view(np.uint16)
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        if r1 == r0:
            continue
        qa_r, sa_r, qb_r, sb_r = ref[g]
        assert np.array_equal(qa[r0:r1].cpu().numpy(), qa_r)
        R, S = oracle.gemm_e4m3(qa_r, qb_r)
        check_bf16_like(bf16_bits_to_f64(h[r0:r1]), R, S, sa_r, sb_r, f"group {g}")


def test_grouped_equals_per_group_calls():
    G, total, N, K = 6, 2000, 768, 1024
    A, B, offs = synth.make_moe_inputs(G, total, N, K, seed=3, empty=1)
    qa, qb, sa, sb, _ = quantise_groups(A, B, offs, N)
    Dg = torch.zeros((total, N), dtype=torch.bfloat16, device="cuda")
    dg.dg_fp8_gemm_grouped(qa, qb, Dg, dev(offs), sa, sb, None, dg.DG_BF16, M=total, N=N, K=K,
                           groups=G)
    Ds = torch.zeros((total, N), dtype=torch.bfloat16, device="cuda")
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        if r1 > r0:
            dg.dg_fp8_gemm(qa[r0:r1], qb[g * N:(g + 1) * N], Ds[r0:r1], sa[g:g + 1], sb[g:g + 1],
                           None, dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    # same FP32 contraction order per tile, so the results agree exactly
    # except where different tile widths change the summation grouping
    a, b = Dg.float(), Ds.float()
    assert torch.allclose(a, b, rtol=1e-2, atol=1e-2 * float(b.abs().max()))


def test_grouped_e4m3_out():
    G, total, N, K = 4, 900, 400, 512
    A, B, offs = synth.make_moe_inputs(G, total, N, K, seed=5)
    qa, qb, sa, sb, ref = quantise_groups(A, B, offs, N)
    sd_host = []
    for g in range(G):
        qa_r, sa_r, qb_r, sb_r = ref[g]
        R = oracle.gemm_e4m3(qa_r, qb_r, with_abs=False)
        sd_host.append(np.float32(np.max(np.abs(oracle.epilogue_scale(R, sa_r, sb_r))) / 448.0))
    sd = dev(np.array(sd_host, np.float32))
    D = torch.empty((total, N), dtype=torch.uint8, device="cuda")
    dg.dg_fp8_gemm_grouped(qa, qb, D, dev(offs), sa, sb, sd, dg.DG_E4M3, M=total, N=N, K=K, groups=G)
    assert dg.dg_sync_status() == dg.DG_OK
    h = D.cpu().numpy()
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        qa_r, sa_r, qb_r, sb_r = ref[g]
        R = oracle.gemm_e4m3(qa_r, qb_r, with_abs=False)
        check_e4m3(h[r0:r1], R, sa_r, sb_r, sd_host[g])


@pytest.mark.parametrize("bad", [[0, 50, 40, 100], [1, 50, 60, 100], [0, 50, 60, 90]])
def test_grouped_invalid_offsets_store_nothing(bad):
    """Decreasing offsets, a non-zero start or an end other than M: the kernel
    stores nothing and the status reports DG_ERR_INVALID_VALUE."""
    total, N, K = 100, 128, 64
    qa = torch.zeros((total, K), dtype=torch.uint8, device="cuda")
    qb = torch.zeros((3 * N, K), dtype=torch.uint8, device="cuda")
    s = torch.ones(3, dtype=torch.float32, device="cuda")
    D = torch.full((total, N), 0x7FFF, dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_grouped(qa, qb, D, dev(np.array(bad, np.int32)), s, s, None, dg.DG_BF16,
                           M=total, N=N, K=K, groups=3)
    assert dg.dg_sync_status() == dg.DG_ERR_INVALID_VALUE
    assert dg.dg_sync_status() == dg.DG_OK
    assert torch.all(D == 0x7FFF)

"""Output-range parity: the ends of the output formats on every kernel path.

[FP8-guide] §4.3 clamps the E4M3 map to +-448 and §3.2 sends the GEMM output
through the same map after the division by the output scale, so with a small
scale_d many outputs saturate, and with a large one they fall into the E4M3
subnormal range (|y| < 2^-6).  [DG-FP16] §3.3 is about FP16 overflow: a sum
beyond 65504 becomes +-Inf when rounded to binary16.  Each case here drives
one kernel (GEMV, split-K, single-CTA tiles, CTA pairs, warp-MMA GEMV,
grouped) into those
ranges and compares every output with the oracle: E4M3 codes within one
step of e4m3(Dref / sD) and exactly +-448 where Dref / sD is clearly beyond
the clamp; FP16 outputs +-Inf exactly where the exact sum is clearly beyond
the binary16 range, and within the usual tolerance elsewhere.
"""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import (REL, ABS, check_e4m3, check_guards, check_quantised, dev, fp16_bits_to_f64,
                     gpu_quantize, guarded, scalar)

pytestmark = pytest.mark.gpu

# (M, N, K, tuning variables, expected plan path, expected block_m)
PATHS = {
    "gemv": (1, 1000, 1040, {"DG_MMA_GEMV": "0"}, 2, None),
    "splitk": (8, 1000, 1040, {"DG_MMA_GEMV": "0"}, 4, 16),
    "single_cta": (129, 1000, 1040, {"DG_2CTA": "0"}, 3, 128),
    "cta_pair": (512, 1000, 1040, {"DG_2CTA": "1"}, 3, 256),
    "gemv_mma": (16, 1000, 1040, {"DG_MMA_GEMV": "1"}, 5, None),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def _expect_plan(M, N, K, path, block_m, in_dtype=dg.DG_E4M3, out=dg.DG_E4M3):
    p = dg.dg_gemm_plan(M, N, K, in_dtype, out)
    assert p["path"] == path, p
    if block_m is not None:
        assert p["block_m"] == block_m, p


def _output_scale(dref, mode):
    """An output scale from the oracle's Dref that puts the median output at
    2 x 448 (`saturate`: about half the outputs clamp) or at 2^-7
    (`subnormal`: about half land below 2^-6).  The median, not the
    maximum, because the workload's outliers make a few outputs large."""
    med = float(np.median(np.abs(dref)))
    return np.float32(med / 896.0) if mode == "saturate" else np.float32(med * 128.0)


def _e4m3_case(M, N, K, mode):
    """GPU quantise + GEMM with E4M3 output at the scale above."""
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa, amax_a, sa = gpu_quantize(A)
    qb, amax_b, sb = gpu_quantize(B)
    qa_ref, sa_ref = check_quantised(A, qa, amax_a, sa)
    qb_ref, sb_ref = check_quantised(B, qb, amax_b, sb)
    R = oracle.gemm_e4m3(qa_ref, qb_ref, with_abs=False)
    sd = _output_scale(oracle.epilogue_scale(R, sa_ref, sb_ref), mode)
    sdt = scalar()
    sdt[0] = float(sd)
    buf, D = guarded(M * N, torch.uint8, 0x7F)
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, sdt, dg.DG_E4M3, M=M, N=N, K=K)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F)
    return D.cpu().numpy().reshape(M, N), R, sa_ref, sb_ref, sd


def _check_range(codes, R, sa, sb, sd, mode):
    check_e4m3(codes, R, sa, sb, sd)
    assert not np.any((codes & 0x7F) == 0x7F), "NaN code in the output"
    y = oracle.epilogue_scale(R, sa, sb) / float(sd)
    ref = oracle.epilogue_e4m3(R, sa, sb, sd)
    if mode == "saturate":
        # far beyond the clamp (464 is the rounding midpoint above 448):
        # exactly +-448, sign kept
        far = np.abs(y) > 480.0
        assert far.sum() > 0.3 * y.size, far.sum()       # the case does saturate
        assert (y[far] < 0).any() and (y[far] > 0).any()
        want = np.where(y[far] > 0, 0x7E, 0xFE)
        assert np.array_equal(codes[far], want), np.flatnonzero(codes[far] != want)[:5]
    else:
        sub = ((ref & 0x78) == 0) & ((ref & 0x07) != 0)   # exponent field 0, non-zero
        assert sub.sum() > 0.3 * y.size, sub.sum()         # the case reaches subnormals


@pytest.mark.parametrize("mode", ["saturate", "subnormal"])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_e4m3_output_saturation_and_subnormals(path, mode):
    M, N, K, kv, want_path, want_bm = PATHS[path]
    with knobs(**kv):
        _expect_plan(M, N, K, want_path, want_bm)
        codes, R, sa, sb, sd = _e4m3_case(M, N, K, mode)
    _check_range(codes, R, sa, sb, sd, mode)


@pytest.mark.parametrize("mode", ["saturate", "subnormal"])
def test_e4m3_output_range_grouped(mode):
    """The grouped kernel (per-group output scales) at both ends."""
    G, N, K = 4, 384, 1040
    A32, B32, offs = synth.make_moe_inputs(G, 700, N, K, seed=11, empty=1)
    M = A32.shape[0]
    qa, amax_a, sa = gpu_quantize(A32)
    qa_ref, sa_ref = check_quantised(A32, qa, amax_a, sa)
    qbs, sbs, refs = [], [], []
    for g in range(G):
        qb, amax_b, sb = gpu_quantize(B32[g * N:(g + 1) * N])
        qbs.append(qb)
        sbs.append(sb[0:1])
        refs.append(check_quantised(B32[g * N:(g + 1) * N], qb, amax_b, sb))
    qb_all = torch.cat(qbs)
    sa_g = torch.cat([sa[0:1]] * G)
    sb_g = torch.cat(sbs)
    Rs, sds = [], []
    for g in range(G):
        rows = slice(offs[g], offs[g + 1])
        R = oracle.gemm_e4m3(qa_ref[rows], refs[g][0], with_abs=False)
        Rs.append(R)
        sds.append(_output_scale(oracle.epilogue_scale(R, sa_ref, refs[g][1]), mode)
                   if R.size else np.float32(1.0))
    sd_g = torch.tensor(np.array(sds, np.float32), device="cuda")
    buf, D = guarded(M * N, torch.uint8, 0x7F)
    doffs = torch.tensor(np.asarray(offs, np.int32), device="cuda")
    dg.dg_fp8_gemm_grouped(qa, qb_all, D, doffs, sa_g, sb_g, sd_g, dg.DG_E4M3, M=M, N=N, K=K,
                           groups=G)
    assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7F)
    h = D.cpu().numpy().reshape(M, N)
    for g in range(G):
        if offs[g + 1] > offs[g]:
            _check_range(h[offs[g]:offs[g + 1]], Rs[g], sa_ref, refs[g][1], sds[g], mode)


# ---------------------------------------------------------------- FP16 overflow

F16_MAX_MID = 65520.0   # halfway between 65504 and the next binade: RNE -> Inf above


def _check_fp16_overflow(d, R, S, sa, sb):
    """+-Inf exactly where |Dref| is clearly past the binary16 range, the
    ordinary tolerance where it is clearly inside, either near the edge."""
    dref = oracle.epilogue_scale(R, sa, sb)
    bound = REL * np.abs(dref) + ABS * S * float(sa) * float(sb)
    over = np.abs(dref) - bound > F16_MAX_MID
    inside = np.abs(dref) + bound < 65504.0
    assert over.sum() > 0.05 * d.size and inside.sum() > 0.05 * d.size, (over.sum(), inside.sum())
    assert np.all(np.isinf(d[over])) and np.all(np.sign(d[over]) == np.sign(dref[over])), \
        np.flatnonzero(~np.isinf(d[over]))[:5]
    err = np.abs(d[inside] - dref[inside])
    bad = np.flatnonzero(~(err <= bound[inside]))
    assert bad.size == 0, (bad[:5], d[inside][bad[:5]], dref[inside][bad[:5]])
    edge = ~over & ~inside
    if edge.any():   # either the nearest finite value or +-Inf of the right sign
        de, re_, be = d[edge], dref[edge], bound[edge]
        ok = (np.isinf(de) & (np.sign(de) == np.sign(re_))) | (np.abs(de - re_) <= be)
        assert ok.all()
    assert not np.isnan(d).any()


@pytest.mark.parametrize("path", sorted(PATHS))
def test_hgemm_fp16_output_overflows_to_inf(path):
    """FP16 operands U(-1,1) x 100: products up to 1e4, sums over K = 1040
    mostly beyond 65504."""
    M, N, K, kv, want_path, want_bm = PATHS[path]
    rng = np.random.default_rng(5)
    A16 = (rng.uniform(-1, 1, (M, K)) * 100).astype(np.float16)
    B16 = (rng.uniform(-1, 1, (N, K)) * 100).astype(np.float16)
    with knobs(**kv):
        _expect_plan(M, N, K, want_path, want_bm, dg.DG_FP16, dg.DG_FP16)
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
        dg.dg_hgemm(dev(A16.view(np.int16)), dev(B16.view(np.int16)), D, dg.DG_FP16, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.hgemm(A16.view(np.uint16), B16.view(np.uint16))
    d = fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N))
    _check_fp16_overflow(d, R, S, 1.0, 1.0)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_fp8_gemm_fp16_output_overflows_to_inf(path):
    """E4M3 GEMM with FP16 output: scale_a * scale_b large enough that most
    outputs leave the binary16 range."""
    M, N, K, kv, want_path, want_bm = PATHS[path]
    A, B = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    qa_ref, _, _ = oracle.quantize_tensor(A)
    qb_ref, _, _ = oracle.quantize_tensor(B)
    s = scalar()
    s[0] = 16.0
    with knobs(**kv):
        _expect_plan(M, N, K, want_path, want_bm, dg.DG_E4M3, dg.DG_FP16)
        buf, D = guarded(M * N, torch.int16, 0x7FFF)
        dg.dg_fp8_gemm(dev(qa_ref), dev(qb_ref), D, s, s, None, dg.DG_FP16, M=M, N=N, K=K)
        assert dg.dg_sync_status() == dg.DG_OK
    check_guards(buf, M * N, 0x7FFF)
    R, S = oracle.gemm_e4m3(qa_ref, qb_ref)
    d = fp16_bits_to_f64(D.cpu().numpy().view(np.uint16).reshape(M, N))
    _check_fp16_overflow(d, R, S, np.float32(16.0), np.float32(16.0))

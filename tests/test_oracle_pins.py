"""Pins for the CPU oracle: facts that the pages and mathematics fix.

Each check is independent of the oracle's own code path (format facts,
worked rounding cases, closed forms, exact rational brute force, an
independent integer contraction and library cross-checks), chosen so that a
dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them.  CPU only.

[FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南" (sheratonhq.com/news/156926).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLDEN, "page_facts.json"), encoding="utf-8"))

ALL = np.arange(256, dtype=np.uint8)
NAN_CODES = {0x7F, 0xFF}


def frac_e4m3(c: int) -> Fraction:
    """Exact value of an E4M3 code, from the bit fields, as a Fraction."""
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    v = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return -v if s else v


# ---------------------------------------------------------------- E4M3 table

def test_e4m3_page_facts():
    tab = oracle.e4m3_decode(ALL)
    assert FACTS["e4m3_max_finite"]["value"] == 448.0
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0
    assert np.nanmax(tab) == 448.0 and np.nanmin(tab) == -448.0
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])
    assert np.isnan(tab).sum() == 2
    assert tab[0x01] == 2.0 ** -9 and tab[0x08] == 2.0 ** -6 and tab[0x38] == 1.0
    assert FACTS["e4m3_bits"]["exponent_bits"] == 4


def test_e4m3_decode_matches_bitfields_exactly():
    tab = oracle.e4m3_decode(ALL)
    for c in range(256):
        if c in NAN_CODES:
            continue
        assert Fraction(tab[c]) == frac_e4m3(c), hex(c)


def test_e4m3_roundtrip_and_monotone():
    tab = oracle.e4m3_decode(ALL)
    for c in range(256):
        if c in NAN_CODES:
            continue
        assert oracle.e4m3_encode(tab[c]) == c, hex(c)
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(tab[0x80:0xFF], -pos)


def test_e4m3_decode_matches_torch():
    t = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).float().numpy()
    tab = oracle.e4m3_decode(ALL)
    assert np.array_equal(np.isnan(t), np.isnan(tab))
    ok = ~np.isnan(tab)
    assert np.array_equal(t[ok].astype(np.float64), tab[ok])


# ------------------------------------------------------------ E4M3 encoder

@pytest.mark.parametrize("y,code", [
    (1.0625, 0x38),          # tie 1.0 | 1.125 -> even mantissa (1.0)
    (1.1875, 0x3A),          # tie 1.125 | 1.25 -> 1.25
    (2.0 ** -10, 0x00),      # tie 0 | 2^-9 -> +0
    (3 * 2.0 ** -10, 0x02),  # tie 2^-9 | 2^-8 -> 2^-8
    (1.9375, 0x40),          # tie across a binade: 1.875 | 2.0 -> 2.0
    (432.0, 0x7E),           # tie 416 | 448 -> 448
    (464.0, 0x7E),           # saturate
    (1e9, 0x7E),
    (-1e9, 0xFE),
    (float("inf"), 0x7E),
    (float("-inf"), 0xFE),
    (-(2.0 ** -11), 0x80),   # negative underflow keeps the sign
    (-0.0, 0x80),
    (0.0, 0x00),
    (1.06, 0x38),
    (1.07, 0x39),
])
def test_e4m3_encode_worked_cases(y, code):
    assert oracle.e4m3_encode(y) == code


def test_e4m3_encode_nan():
    assert oracle.e4m3_encode(float("nan")) in (0x7F, 0xFF)


def test_e4m3_encode_matches_torch_in_range():
    rng_vals = synth.normal_f32(11, (20000,)) * np.float32(64.0)
    tab = oracle.e4m3_decode(ALL)
    fin = tab[~np.isnan(tab)]
    fin = np.sort(fin)
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)   # every tie point
    eps = np.float32(2.0 ** -20)
    vals = np.concatenate([rng_vals, mids, mids * (1 + eps), mids * (1 - eps),
                           fin.astype(np.float32)])
    vals = vals[np.abs(vals) <= 448]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(vals.astype(np.float64))
    assert np.array_equal(got, ref)


# ---------------------------------------------------------- other formats

def test_fp16_decode_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.fp16_decode(bits)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_bf16_decode_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = oracle.bf16_decode(bits)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_bf16_encode_matches_torch():
    v = np.concatenate([
        synth.normal_f32(5, (30000,)) * np.float32(1e3),
        np.float32([0.0, -0.0, 1.0, 3.0e38, -3.3e38, 1e-40, -1e-41, 1.00390625,
                    1.01171875, np.inf, -np.inf]),
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_encode(v)
    assert np.array_equal(got, ref)


def test_fp16_encode_matches_numpy():
    v = np.concatenate([synth.normal(6, 30000) * 100.0,
                        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -25,
                         3 * 2.0 ** -26, -1e6]])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = oracle.fp16_encode(v)
    assert np.array_equal(got, ref)


# ----------------------------------------------------- amax, scale, quantiser

def test_amax_and_scale():
    x = synth.normal_f32(3, (1000, 37))
    a = oracle.amax(x)
    assert a == np.max(np.abs(x))
    s = oracle.scale_from_amax(a)
    assert FACTS["scale_rule"]["divisor"] == 448.0
    # s is the binary32 value nearest amax/448: amax lies within half an ulp
    # of s*448 in exact arithmetic
    err = abs(Fraction(float(s)) * 448 - Fraction(float(a)))
    assert err <= Fraction(float(np.spacing(s))) * 448 / 2
    assert oracle.scale_from_amax(0.0) == 1.0
    y = x.copy()
    y[5, 5] = np.nan
    assert np.isnan(oracle.amax(y))
    assert oracle.amax(np.float32([-3.0, 2.0])) == 3.0


def test_quantiser_matches_torch_reference_path():
    """Independent path: torch CPU float32 divide, clamp, RNE cast."""
    A, B = synth.make_inputs("fp8_sweep_m65")
    for x in (A, B, synth.normal_f32(9, (4096,)) * np.float32(1e-3)):
        q, s, a = oracle.quantize_tensor(x)
        t = torch.from_numpy(x) / torch.tensor(s, dtype=torch.float32)
        ref = t.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q, ref)
        # the largest-magnitude element lands exactly on +-448
        i = np.argmax(np.abs(x))
        assert q.reshape(-1)[i] in (0x7E, 0xFE)


def test_quantiser_random_scales_match_torch():
    x = synth.normal_f32(12, (50000,)) * np.float32(30.0)
    for k, s in enumerate([1.0, 0.37, 3.0e-3, 1.7e4, 2.0 ** -20]):
        q = oracle.quantize_e4m3(x, np.float32(s))
        t = torch.from_numpy(x) / torch.tensor(np.float32(s))
        ref = t.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q, ref), k


def test_quantiser_special_values():
    x = np.float32([np.inf, -np.inf, 0.0, -0.0, 1e30, -1e30, 1e-30, np.nan])
    q = oracle.quantize_e4m3(x, np.float32(1.0))
    assert list(q[:7]) == [0x7E, 0xFE, 0x00, 0x80, 0x7E, 0xFE, 0x00]
    assert q[7] in (0x7F, 0xFF)


# ------------------------------------------------------------- contractions

def _random_codes(seed, shape):
    c = synth.random_bytes(seed, shape)
    c[(c & 0x7F) == 0x7F] = 0x38       # drop NaN codes
    return c


@pytest.mark.parametrize("M,N,K", [(4, 4, 4), (3, 5, 16), (7, 9, 1040), (1, 13, 300)])
def test_gemm_equals_independent_integer_sum(M, N, K):
    A = _random_codes(20 + M, (M, K))
    B = _random_codes(40 + N, (N, K))
    R, S = oracle.gemm_e4m3(A, B)
    units = oracle.gemm_e4m3_exact_units(A, B)
    assert np.array_equal(R, units.astype(np.float64) * 2.0 ** -18)
    assert np.all(S >= np.abs(R))


def test_gemm_bruteforce_4x4x4_fractions():
    A = _random_codes(1, (4, 4))
    B = _random_codes(2, (4, 4))
    R, S = oracle.gemm_e4m3(A, B)
    for m in range(4):
        for n in range(4):
            terms = [frac_e4m3(int(A[m, k])) * frac_e4m3(int(B[n, k])) for k in range(4)]
            assert Fraction(R[m, n]) == sum(terms)
            assert Fraction(S[m, n]) == sum(abs(t) for t in terms)


def test_gemm_matches_library_matmul():
    """FP64 matmul of the decoded operands is exact here (every partial sum
    is a multiple of 2^-18 below 2^53), so it must agree bit for bit."""
    A = _random_codes(3, (33, 517))
    B = _random_codes(4, (65, 517))
    R = oracle.gemm_e4m3(A, B, with_abs=False)
    ref = oracle.e4m3_decode(A) @ oracle.e4m3_decode(B).T
    assert np.array_equal(R, ref)


def test_gemm_closed_forms():
    K = 48
    one = 0x38
    # identity: R = dec(B)^T, which also fixes the operand orientation
    A = np.zeros((K, K), np.uint8)
    np.fill_diagonal(A, one)
    B = _random_codes(5, (20, K))
    R = oracle.gemm_e4m3(A, B, with_abs=False)
    assert np.array_equal(R, oracle.e4m3_decode(B).T)
    # one-hot rows pick single columns of B, scaled by the hot value
    A = np.zeros((3, K), np.uint8)
    A[0, 7] = 0x40      # 2.0
    A[1, 0] = 0xB8      # -1.0
    A[2, K - 1] = 0x7E  # 448
    R = oracle.gemm_e4m3(A, B, with_abs=False)
    dB = oracle.e4m3_decode(B)
    assert np.array_equal(R[0], 2.0 * dB[:, 7])
    assert np.array_equal(R[1], -dB[:, 0])
    assert np.array_equal(R[2], 448.0 * dB[:, K - 1])
    # zero operand
    R = oracle.gemm_e4m3(np.zeros((2, K), np.uint8), B, with_abs=False)
    assert np.all(R == 0)


def test_all_ones_gives_k_page_worked_check():
    """[FP8-guide] §5.4: all-ones inputs must give K everywhere, also through
    the full per-tensor quantise -> GEMM -> scale chain."""
    for K in (1, 16, 1040, 4096):
        x = np.ones((3, K), np.float32)
        qa, sa, _ = oracle.quantize_tensor(x)
        qb, sb, _ = oracle.quantize_tensor(np.ones((5, K), np.float32))
        assert np.all(qa == 0x7E) and np.all(qb == 0x7E)
        R = oracle.gemm_e4m3(qa, qb, with_abs=False)
        assert np.all(R == K * 448.0 * 448.0)
        D = oracle.epilogue_scale(R, sa, sb)
        # sa = sb = fl32(1/448): D = K within two binary32 ulps of the scale
        assert np.all(np.abs(D - K) <= K * 2 * 2.0 ** -23)


def test_quantisation_error_within_page_guidance():
    """[FP8-guide] §4.3: against the unquantised product of random matrices
    a per-tensor E4M3 GEMM lands at a few percent relative error; above 10%
    means a wrong scale.  A multiply-instead-of-divide scale, a dropped
    scale or a transposed operand all blow far past that."""
    A = synth.normal_f32(30, (64, 4096))
    B = synth.normal_f32(31, (96, 4096))
    qa, sa, _ = oracle.quantize_tensor(A)
    qb, sb, _ = oracle.quantize_tensor(B)
    D = oracle.epilogue_scale(oracle.gemm_e4m3(qa, qb, with_abs=False), sa, sb)
    exact = A.astype(np.float64) @ B.astype(np.float64).T
    rel = np.linalg.norm(D - exact) / np.linalg.norm(exact)
    assert 1e-3 < rel < FACTS["quantisation_error_guide"]["wrong_above_rel"]


def test_epilogue_e4m3_out():
    R = np.array([0.0, 1.0, -3.0, 1e9, 5.0, 0.1], np.float64)
    e = oracle.epilogue_e4m3(R, 1.0, 1.0, 1.0)
    assert list(e) == [oracle.e4m3_encode(v) for v in R]
    # power-of-two scales are exact: R*0.5*4/2 == R
    e2 = oracle.epilogue_e4m3(R, 0.5, 4.0, 2.0)
    assert np.array_equal(e, e2)
    # divide by the output scale: 448 * sD -> 448
    assert oracle.epilogue_e4m3(np.array([448.0 * 3.0]), 1.0, 1.0, 3.0)[0] == 0x7E


def test_hgemm_against_fractions_and_library():
    A, B = synth.make_inputs("fp16_4096", M=5, N=6, K=64)
    R, S = oracle.hgemm(A, B)
    dA = A.view(np.float16).astype(np.float64)
    dB = B.view(np.float16).astype(np.float64)
    for m in range(5):
        for n in range(6):
            exact = sum(Fraction(float(dA[m, k])) * Fraction(float(dB[n, k])) for k in range(64))
            assert abs(Fraction(R[m, n]) - exact) <= Fraction(S[m, n]) * Fraction(2) ** -50
    assert np.allclose(R, dA @ dB.T, rtol=0, atol=1e-12)
    r2, s2 = oracle.hgemm_at(A, B, np.array([4, 0]), np.array([1, 5]))
    assert r2[0] == R[4, 1] and r2[1] == R[0, 5] and s2[0] == S[4, 1]


def test_sampled_equals_full():
    A = _random_codes(7, (9, 300))
    B = _random_codes(8, (11, 300))
    R, S = oracle.gemm_e4m3(A, B)
    ms = np.array([0, 8, 3, 8])
    ns = np.array([10, 0, 5, 10])
    r, s = oracle.gemm_e4m3_at(A, B, ms, ns)
    assert np.array_equal(r, R[ms, ns]) and np.array_equal(s, S[ms, ns])


def test_threading_does_not_change_results():
    A = _random_codes(9, (17, 200))
    B = _random_codes(10, (23, 200))
    R1 = oracle.gemm_e4m3(A, B, with_abs=False, nthreads=1)
    R7 = oracle.gemm_e4m3(A, B, with_abs=False, nthreads=7)
    assert np.array_equal(R1, R7)


def test_tolerance_is_sound_for_bf16_and_fp16_rounding():
    """The oracle's own correctly rounded BF16/FP16 outputs pass the parity
    bound |D - ref| <= 8e-3 |ref| + 1e-4 * S * sA * sB."""
    A, B = synth.make_inputs("fp8_sweep_m63")
    qa, sa, _ = oracle.quantize_tensor(A[:8])
    qb, sb, _ = oracle.quantize_tensor(B[:50])
    R, S = oracle.gemm_e4m3(qa, qb)
    dref = oracle.epilogue_scale(R, sa, sb)
    d = oracle.bf16_decode(oracle.bf16_encode(dref.astype(np.float32)))
    bound = 8e-3 * np.abs(dref) + 1e-4 * S * float(sa) * float(sb)
    assert np.all(np.abs(d - dref) <= bound)
    h = oracle.fp16_decode(oracle.fp16_encode(dref))
    assert np.all(np.abs(h - dref) <= bound)


def test_generator_is_deterministic_and_distributed():
    a = synth.normal(0, 5000)
    b = synth.normal(0, 12000)[:5000]
    assert np.array_equal(a, b)
    z = synth.normal(0, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    A, B = synth.make_inputs("fp8_qkv", N=256)
    assert A.shape == (1, 4096) and B.shape == (256, 4096)
    assert abs(float(B.std()) - 0.02) < 0.001
    A, B = synth.make_inputs("fp8_sweep_m1")
    frac = np.mean(np.abs(np.concatenate([A.ravel(), B.ravel()])) > 6.0)
    assert 0.0003 < frac < 0.002   # the 0.1% outliers times 50


# ------------------------------------------------------- power-of-two scale

@pytest.mark.parametrize("amax,scale", [
    (448.0, 1.0),            # exactly the top of the range
    (449.0, 2.0),
    (224.0, 0.5),
    (224.0001, 1.0),
    (1.0, 2.0 ** -8),        # 448 * 2^-9 = 0.875 < 1 <= 448 * 2^-8
    (0.875, 2.0 ** -9),
    (3.0e38, 2.0 ** 120),    # 448 * 2^119 ~ 2.98e38 < 3e38
    (1e-45, 2.0 ** -149),    # clamps at the smallest binary32 power of two
    (0.0, 1.0),
])
def test_pow2_scale_worked_cases(amax, scale):
    assert oracle.scale_pow2_from_amax(amax) == np.float32(scale)


def test_pow2_scale_properties():
    """448 p >= amax > 224 p for every normal amax: the tensor's largest value
    lands in (224, 448] and never saturates; division by p is exact."""
    a = np.abs(synth.normal_f32(40, (5000,)) * np.float32(1e3)) + np.float32(1e-3)
    for v in a[:500]:
        p = float(oracle.scale_pow2_from_amax(v))
        assert np.log2(p) == int(np.log2(p))
        assert 448.0 * p >= float(v) > 224.0 * p
    assert np.isnan(oracle.scale_pow2_from_amax(np.nan))
    assert np.isinf(oracle.scale_pow2_from_amax(np.inf))
    x = synth.normal_f32(41, (4096,))
    q, s, am = oracle.quantize_tensor_pow2(x)
    # division by a power of two is exact, so quantising x/p equals encoding x*2^-e
    ref = oracle.e4m3_encode(x.astype(np.float64) / float(s))
    assert np.array_equal(q, ref)
    assert np.max(q & 0x7F) <= 0x7E


def test_pow2_scale_accuracy_against_amax_scale():
    """Accuracy of the chain with the power-of-two scale compared with the
    amax/448 scale on the same inputs ([FP8-guide] §2.1 vs §3.2): both stay
    inside the page's 10% bound; the power of two uses at most one binade
    less of the E4M3 range, so its error is at most about twice as large."""
    A = synth.normal_f32(42, (48, 2048))
    B = synth.normal_f32(43, (64, 2048))
    exact = A.astype(np.float64) @ B.astype(np.float64).T
    errs = []
    for qt in (oracle.quantize_tensor, oracle.quantize_tensor_pow2):
        qa, sa, _ = qt(A)
        qb, sb, _ = qt(B)
        D = oracle.epilogue_scale(oracle.gemm_e4m3(qa, qb, with_abs=False), sa, sb)
        errs.append(np.linalg.norm(D - exact) / np.linalg.norm(exact))
    assert all(e < FACTS["quantisation_error_guide"]["wrong_above_rel"] for e in errs)
    assert errs[1] <= 2.5 * errs[0]


# ---------------------------------------------------------------------------
# FP16 dynamic-range scaling ([DG-FP16] §3.3): scale = min(1, 65504 /
# (max|A| max|B|)); A, B times sqrt(scale) into FP16; result divided by scale.

def _is_correctly_rounded_f32(r, exact):
    """r (float32) is the binary32 value nearest to the rational `exact`."""
    from fractions import Fraction
    r = np.float32(r)
    lo = np.nextafter(r, np.float32(-np.inf))
    hi = np.nextafter(r, np.float32(np.inf))
    fr = Fraction(float(r))
    return (abs(Fraction(float(lo)) - exact) >= abs(fr - exact) and
            abs(Fraction(float(hi)) - exact) >= abs(fr - exact))


def test_fp16_range_scale_closed_forms():
    f = oracle.fp16_range_scale
    assert list(f(1.0, 1.0)) == [1, 1, 1, 1]
    assert list(f(256.0, 255.875)) == [1, 1, 1, 1]              # product exactly 65504
    s = f(256.0, 256.0)                                         # 65504 / 65536
    assert s[0] == np.float32(1 - 2 ** -11)
    s = f(1024.0, 1024.0)                                       # 65504 / 2^20, exact
    assert s[0] == np.float32(65504 / 2 ** 20)
    assert list(f(0.0, 7.0)) == [1, 1, 1, 1]                    # all-zero operand
    assert np.isnan(f(np.nan, 1.0)[0]) and np.isnan(f(1.0, np.nan)[0])
    assert f(3e38, 3e38)[0] == np.float32(65504 / 9e76)        # product formed in FP64
    assert f(1e6, 1e6)[3] == 1.0


def test_fp16_range_scale_sqrt_and_reciprocal_correctly_rounded():
    from fractions import Fraction
    rng = np.random.default_rng(5)
    for a, b in zip(10 ** rng.uniform(-3, 12, 300), 10 ** rng.uniform(-3, 12, 300)):
        s, r, inv, one = oracle.fp16_range_scale(np.float32(a), np.float32(b))
        exact_s = min(Fraction(1), Fraction(65504) / (Fraction(float(np.float32(a))) *
                                                      Fraction(float(np.float32(b)))))
        assert _is_correctly_rounded_f32(s, exact_s)
        assert 0 < s <= 1 and one == 1
        # sqrt: r is the float nearest to sqrt(s), i.e. the midpoints around r
        # bracket s when squared
        rs = Fraction(float(r))
        lo = (rs + Fraction(float(np.nextafter(r, np.float32(0))))) / 2
        hi = (rs + Fraction(float(np.nextafter(r, np.float32(2))))) / 2
        assert lo * lo <= Fraction(float(s)) <= hi * hi
        assert _is_correctly_rounded_f32(inv, 1 / Fraction(float(s)))


def test_convert_f16_matches_numpy_half_cast():
    """fp16_rn(fl32(x * factor)) against numpy's binary32 multiply and
    binary32 -> binary16 cast (round to nearest even, overflow to Inf)."""
    rng = np.random.default_rng(6)
    x = np.concatenate([
        (rng.standard_normal(20000) * 10 ** rng.uniform(-9, 6, 20000)).astype(np.float32),
        np.float32([0.0, -0.0, 1.0, 65504, 65519.99, 65520, -65520, 1e9, np.inf, -np.inf,
                    2 ** -24, 2 ** -25, 3 * 2 ** -26, 2 ** -14, 1 + 2 ** -11, 1 + 3 * 2 ** -11]),
    ])
    for factor in (1.0, 0.24993895, 3.5, 2 ** -7):
        got = oracle.convert_f16(x, factor)
        with np.errstate(over="ignore"):
            want = (x * np.float32(factor)).astype(np.float16).view(np.uint16)
        assert np.array_equal(got, want), factor
    nan = oracle.convert_f16(np.float32([np.nan]), 1.0)
    assert (nan[0] & 0x7C00) == 0x7C00 and (nan[0] & 0x03FF) != 0


def test_fp16_range_chain_recovers_out_of_range_product():
    """A holds outliers far beyond FP16 (so plain conversion gives Inf); the
    scaled chain reproduces the FP64 product of the original FP32 operands
    within the FP16 rounding of each operand: |Delta x| <= |x| (2^-11 + 2^-24)
    + 2^-25 / sqrt(scale), and the binary32 rounding of sqrt(scale) and 1/scale."""
    M, N, K = 6, 40, 96
    A, B = synth.make_inputs("fp8_256", M=M, N=N, K=K)
    A = A.copy()
    A[1, 5] = 9.0e4
    A[4, 17] = -7.5e4
    A[0, 0] = 7.0e4
    assert (oracle.convert_f16(A, 1.0) & 0x7FFF).max() == 0x7C00     # plain cast overflows
    f, A16, B16, D, S = oracle.fp16_range_chain(A, B)
    assert f[0] < 1
    assert np.all(np.isfinite(oracle.fp16_decode(A16)))
    exact = A.astype(np.float64) @ B.astype(np.float64).T
    r = float(f[1])
    ea = np.abs(A.astype(np.float64)) * (2 ** -11 + 2 ** -24) + 2 ** -25 / r
    eb = np.abs(B.astype(np.float64)) * (2 ** -11 + 2 ** -24) + 2 ** -25 / r
    bound = (ea @ np.abs(B.astype(np.float64)).T + np.abs(A.astype(np.float64)) @ eb.T + ea @ eb.T)
    bound = bound * (1 + 2 ** -20) + 2 ** -20 * np.abs(exact)
    assert np.all(np.abs(D - exact) <= bound)
    # dropping the final division by scale is caught
    assert not np.all(np.abs(D * float(f[0]) - exact) <= bound)


def test_fp16_range_scale_bounds_products_not_operands():
    """The page's single scale keeps every |a b| scale within 65504; one
    operand alone still overflows once max|A| / max|B| exceeds 65504."""
    f = oracle.fp16_range_scale(9.0e5, 4.0)
    assert np.float64(9.0e5) * 4.0 * float(f[0]) <= 65504 * (1 + 2 ** -23)
    assert oracle.convert_f16(np.float32([9.0e5]), f[1])[0] == 0x7C00          # +Inf
    g = oracle.fp16_range_scale(6.0e4, 1.0)                                     # ratio < 65504
    assert oracle.convert_f16(np.float32([6.0e4]), g[1])[0] != 0x7C00

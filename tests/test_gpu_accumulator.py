"""Is the tensor-core accumulation FP32?  Designed inputs with exact answers.

[FP8-guide] §2.1 (and [HGEMM-L2] §1.3 for FP16 inputs) fix the accumulator
at FP32.  Random inputs cannot show a narrower one: the 1e-4 * S term of
the tolerance hides an accumulator of about 13 bits.  Here every output
holds one large product P = a0 * b0 at the first k, many small products p
after it, and -P at the last k, so the running sum sits near P while the
small products arrive and the exact result is (count of small products) *
p.  The values are chosen so that P + j * p is exactly representable in
binary32 for every j (p is a multiple of the binary32 spacing at P, and
every partial sum stays below the next power of two): FP32 accumulation in
ANY order and grouping returns the exact result, while an accumulator that
keeps fewer bits than FP32 next to P loses the small products outright.
The exact results are powers of two times p, so the BF16 / FP16 outputs
represent them exactly and the check is equality.

Cases, for E4M3 inputs (kind::f8f6f4 MMA, 32 K elements per instruction)
and FP16 inputs (kind::f16, 16 per instruction):
  * across instructions: P at k = 0, -P at k = K - 1, the small products
    in between, spread over many MMA instructions and K blocks;
  * within one instruction: P, the small products and -P inside one
    instruction's K window.
Each runs on the GEMV, split-K (16 and 64 columns), single-CTA, CTA-pair
and warp-MMA GEMV kernels.  The E4M3 cases also read max |acc| back in binary32 through
dg_fp8_gemm_amax, which must equal the exact largest output.
"""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
from _knobs import knobs
from _parity import bf16_bits_to_f64, dev, fp16_bits_to_f64, scalar

pytestmark = pytest.mark.gpu

# E4M3 codes from the format (bias 7, 3 mantissa bits): sign | exponent | mantissa
E4_448 = 0b0_1111_110      # 1.75 * 2^8
E4_QUARTER = 0b0_0101_000  # 2^-2
E4_EIGHTH = 0b0_0100_000   # 2^-3
NEG = 0x80
# binary16 bit patterns
F16_2048 = 0x6800          # 2^11
F16_ONE = 0x3C00
F16_HALF = 0x3800
F16_NEG = 0x8000

# (M, N, tuning variables, expected path, expected block_m)
KERNELS = {
    "gemv": (1, 1000, {"DG_MMA_GEMV": "0"}, 2, None),
    "splitk16": (8, 1000, {"DG_MMA_GEMV": "0"}, 4, 16),
    "splitk64": (64, 1000, {"DG_SPLITK": "1"}, 4, 64),
    "single_cta": (129, 1000, {"DG_2CTA": "0"}, 3, 128),
    "cta_pair": (512, 1000, {"DG_2CTA": "1"}, 3, 256),
    "gemv_mma1": (1, 1000, {"DG_MMA_GEMV": "1"}, 5, None),
    "gemv_mma16": (16, 1000, {"DG_MMA_GEMV": "1"}, 5, None),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def test_codes_mean_what_the_design_says():
    assert oracle.e4m3_decode(np.uint8([E4_448, E4_448 | NEG, E4_QUARTER, E4_EIGHTH])).tolist() == \
        [448.0, -448.0, 0.25, 0.125]
    assert oracle.fp16_decode(np.uint16([F16_2048, F16_2048 | F16_NEG, F16_ONE, F16_HALF])).tolist() == \
        [2048.0, -2048.0, 1.0, 0.5]


def _counts(rows, offset, mult, limit):
    """Small products per row: powers of two 1 .. limit, row 0 with `limit`
    when offset is 0 (a different mix per row; exact in every output format)."""
    top = int(np.log2(limit))
    return np.array([1 << (top - (mult * r + offset) % (top + 1)) for r in range(rows)], np.int64)


def _design(M, N, K, big, neg_big, small_a, small_b, window, dtype):
    """A (M x K) and B (N x K) with big at k0, small products at k0+1 ..,
    big / -big at k0 + window - 1; rows get different small-product counts,
    so D[m, n] = min(cm[m], cn[n]) * p."""
    k0 = 0 if window == K else (K // 2) // window * window   # an instruction-aligned window
    limit = 4096 if window == K else window - 2
    limit = 1 << int(np.log2(min(limit, window - 2)))
    cm = _counts(M, 0, 1, limit)
    cn = _counts(N, 1, 3, limit)
    A = np.zeros((M, K), dtype)
    B = np.zeros((N, K), dtype)
    A[:, k0] = big
    B[:, k0] = big
    A[:, k0 + window - 1] = big
    B[:, k0 + window - 1] = neg_big
    for m in range(M):
        A[m, k0 + 1:k0 + 1 + cm[m]] = small_a
    for n in range(N):
        B[n, k0 + 1:k0 + 1 + cn[n]] = small_b
    return A, B, np.minimum(cm[:, None], cn[None, :]).astype(np.float64)


def _report(got, exact, S, what):
    err = np.abs(got - exact)
    bad = np.flatnonzero(err != 0)
    ratio = float(np.max(err / S)) if err.size else 0.0
    assert bad.size == 0, (f"{what}: {bad.size}/{err.size} outputs differ from the exact sum; "
                           f"max |D - Dref| = {err.max():.6g}, max |D - Dref| / S = {ratio:.3g}; "
                           f"first {bad[:4]} got {got.reshape(-1)[bad[:4]]} "
                           f"want {exact.reshape(-1)[bad[:4]]}")


@pytest.mark.parametrize("case", ["across", "within"])
@pytest.mark.parametrize("small", ["quarter", "eighth"])
@pytest.mark.parametrize("kern", sorted(KERNELS))
def test_e4m3_accumulation_is_fp32(kern, small, case):
    """P = 448 * 448 = 200704 (binary32 spacing 2^-6 there); p = 2^-4
    (0.25 * 0.25) or 2^-6 (0.125 * 0.125)."""
    M, N, kv, path, bm = KERNELS[kern]
    K = 8192 if case == "across" else 4096
    window = K if case == "across" else 32
    x = E4_QUARTER if small == "quarter" else E4_EIGHTH
    p = 2.0 ** -4 if small == "quarter" else 2.0 ** -6
    A, B, cnt = _design(M, N, K, E4_448, E4_448 | NEG, x, x, window, np.uint8)
    exact = cnt * p
    R, S = oracle.gemm_e4m3(A, B)
    assert np.array_equal(R, exact)            # the design is what the docstring says
    one = scalar()
    one[0] = 1.0
    with knobs(**kv):
        plan = dg.dg_gemm_plan(M, N, K, dg.DG_E4M3, dg.DG_BF16)
        assert plan["path"] == path and (bm is None or plan["block_m"] == bm), plan
        D = torch.empty((M, N), dtype=torch.int16, device="cuda")
        am = scalar()
        dg.dg_fp8_gemm_amax(dev(A), dev(B), D, one, one, None, dg.DG_BF16, am)
        assert dg.dg_sync_status() == dg.DG_OK
    got = bf16_bits_to_f64(D.cpu().numpy().view(np.uint16))
    _report(got, exact, S, f"E4M3 {kern} {case} p={p}")
    assert am[0].item() == exact.max(), (am[0].item(), exact.max())   # binary32 readout


@pytest.mark.parametrize("case", ["across", "within"])
@pytest.mark.parametrize("kern", sorted(KERNELS))
def test_fp16_accumulation_is_fp32(kern, case):
    """P = 2048 * 2048 = 2^22 (binary32 spacing 2^-1 there); p = 1 * 0.5."""
    M, N, kv, path, bm = KERNELS[kern]
    K = 4096 if case == "across" else 2048
    window = K if case == "across" else 16
    A, B, cnt = _design(M, N, K, F16_2048, F16_2048 | F16_NEG, F16_ONE, F16_HALF, window,
                        np.uint16)
    exact = cnt * 0.5
    R, S = oracle.hgemm(A, B)
    assert np.array_equal(R, exact)
    with knobs(**kv):
        plan = dg.dg_gemm_plan(M, N, K, dg.DG_FP16, dg.DG_FP16)
        assert plan["path"] == path and (bm is None or plan["block_m"] == bm), plan
        D = torch.empty((M, N), dtype=torch.int16, device="cuda")
        dg.dg_hgemm(dev(A.view(np.int16)), dev(B.view(np.int16)), D, dg.DG_FP16)
        assert dg.dg_sync_status() == dg.DG_OK
    got = fp16_bits_to_f64(D.cpu().numpy().view(np.uint16))
    _report(got, exact, S, f"FP16 {kern} {case}")

"""FP16 dynamic-range scaling on the GPU ([DG-FP16] = the DeepGEMM FP16/WMMA
deep-dive page, §3.3): dg_amax of A and B, dg_fp16_range_scale, dg_convert_f16
of both operands with sqrt(scale), dg_hgemm_scaled with 1/scale.  The
factors and the FP16 operands are bit-exact against the oracle; the GEMM is
within the parity bound of the oracle's exact product of those operands."""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth
from _knobs import knobs
from _parity import bf16_bits_to_f64, check_bf16_like, dev, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def gpu_factors(a, b):
    da, db = dev(np.float32([a, 0, 0, 0])), dev(np.float32([b, 0, 0, 0]))
    f = scalar()
    dg.dg_fp16_range_scale(da, db, f)
    assert dg.dg_sync_status() == dg.DG_OK
    return f.cpu().numpy()


def test_factors_bit_exact():
    rng = np.random.default_rng(8)
    pairs = [(1.0, 1.0), (256.0, 255.875), (256.0, 256.0), (1024.0, 1024.0), (0.0, 3.0),
             (3e38, 3e38), (9.0e5, 4.0), (7.0e4, 3.9)]
    pairs += list(zip(10 ** rng.uniform(-4, 14, 200), 10 ** rng.uniform(-4, 14, 200)))
    for a, b in pairs:
        got = gpu_factors(np.float32(a), np.float32(b))
        want = oracle.fp16_range_scale(np.float32(a), np.float32(b))
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (a, b, got, want)
    got = gpu_factors(np.nan, 1.0)
    assert np.isnan(got[0]) and np.isnan(got[1]) and np.isnan(got[2]) and got[3] == 1


@pytest.mark.parametrize("n", [1, 511, 512, 513, 4096 * 3 + 17, 1 << 20])
def test_convert_bit_exact(n):
    x = (synth.normal_f32(11, (n,)) * np.float32(3e3)).astype(np.float32)
    for factor in (1.0, 0.24993895, 37.0):
        f = dev(np.float32([factor, 0, 0, 0]))
        out = torch.empty(n, dtype=torch.int16, device="cuda")
        dg.dg_convert_f16(dev(x), out, f)
        assert dg.dg_sync_status() == dg.DG_OK
        got = out.cpu().numpy().view(np.uint16)
        assert np.array_equal(got, oracle.convert_f16(x, factor)), (n, factor)


def test_convert_special_values():
    x = np.float32([0.0, -0.0, 65504, 65519.99, 65520, -65520, 1e30, -np.inf, np.inf,
                    2 ** -24, 2 ** -25, 3 * 2 ** -26, 1 + 2 ** -11, 1 + 3 * 2 ** -11, np.nan, 7])
    out = torch.empty(x.size, dtype=torch.int16, device="cuda")
    dg.dg_convert_f16(dev(x), out)       # factor NULL = 1
    assert dg.dg_sync_status() == dg.DG_OK
    got = out.cpu().numpy().view(np.uint16)
    want = oracle.convert_f16(x, 1.0)
    is_nan = lambda h: ((h & 0x7C00) == 0x7C00) & ((h & 0x03FF) != 0)  # noqa: E731
    assert np.array_equal(is_nan(got), is_nan(want))
    assert np.array_equal(got[~is_nan(want)], want[~is_nan(want)])


@pytest.mark.parametrize("M,N,K,mma", [(2, 300, 512, "0"), (9, 1000, 1040, "0"), (2, 300, 512, None),
                                       (9, 1000, 1040, None), (129, 520, 1040, None),
                                       (384, 1000, 2048, None)])
def test_range_scaled_hgemm_chain(M, N, K, mma):
    """Operands with FP16-overflowing outliers: the whole chain on the GPU
    against the oracle's chain (CUDA-core GEMV and split-K with the warp-MMA
    path off, warp-MMA GEMV, single-CTA and pair paths)."""
    with knobs(DG_MMA_GEMV=mma):
        _range_chain(M, N, K)


def _range_chain(M, N, K):
    A, B = synth.make_inputs("fp8_256", M=M, N=N, K=K)
    A = A.copy()
    A[0, 3] = 9.0e4
    A[M - 1, K - 1] = -7.0e4
    dA, dB = dev(A), dev(B)
    am_a, am_b, f = scalar(), scalar(), scalar()
    dg.dg_amax(dA, am_a)
    dg.dg_amax(dB, am_b)
    dg.dg_fp16_range_scale(am_a, am_b, f)
    A16 = torch.empty((M, K), dtype=torch.int16, device="cuda")
    B16 = torch.empty((N, K), dtype=torch.int16, device="cuda")
    dg.dg_convert_f16(dA, A16, f[1:2])
    dg.dg_convert_f16(dB, B16, f[1:2])
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_hgemm_scaled(A16, B16, D, f[2:3], f[3:4], dg.DG_BF16)
    assert dg.dg_sync_status() == dg.DG_OK
    fr, A16r, B16r, Dr, S = oracle.fp16_range_chain(A, B)
    assert np.array_equal(f.cpu().numpy().view(np.uint32), fr.view(np.uint32))
    assert np.array_equal(A16.cpu().numpy().view(np.uint16), A16r)
    assert np.array_equal(B16.cpu().numpy().view(np.uint16), B16r)
    R, _ = oracle.hgemm(A16r, B16r)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S,
                    float(fr[2]), 1.0, "range-scaled HGEMM")
    assert np.all(np.isfinite(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16))))


@pytest.mark.parametrize("n", [0, 1, 511, 512, 4097, (1 << 20) + 7])
def test_convert_with_amax_is_bit_exact(n):
    """The fused pass: codes identical to dg_convert_f16 (and the oracle) and
    the maximum identical to dg_amax (and the oracle), ragged tails included."""
    x = synth.normal_f32(60 + n % 89, (n,)) * np.float32(700.0)
    if n > 10:
        x[7] = -9.5e4             # overflows FP16 at factor 1
    f = scalar()
    f[0] = 0.37
    out = torch.empty(max(n, 1), dtype=torch.int16, device="cuda")[:n]
    am = scalar()
    am[0] = 5.0e6                 # stale: the call zeroes it first
    dg.dg_convert_f16_amax(dev(x), out, f[0:1], am)
    assert dg.dg_sync_status() == dg.DG_OK
    want = oracle.convert_f16(x, np.float32(0.37))
    assert np.array_equal(out.cpu().numpy().view(np.uint16), want)
    assert np.float32(am[0].item()).view(np.uint32) == np.float32(oracle.amax(x)).view(np.uint32)


@pytest.mark.parametrize("na,nb", [(0, 0), (0, 1000), (511, 0), (100, 77), (4097, (1 << 20) + 7),
                                   (1 << 20, 1 << 20)])
def test_convert_pair_is_bit_exact(na, nb):
    """Both operands in one pass: each tensor's codes and maximum identical to
    the oracle (and to dg_convert_f16_amax), ragged tails in the same or in
    different CTAs, empty tensors, stale maxima overwritten."""
    xa = synth.normal_f32(70 + na % 13, (na,)) * np.float32(500.0)
    xb = synth.normal_f32(80 + nb % 17, (nb,)) * np.float32(900.0)
    if na > 10:
        xa[3] = 8.5e4
    if nb > 10:
        xb[nb - 2] = -7.5e4
    f = scalar()
    f[0] = 0.61
    oa = torch.empty(max(na, 1), dtype=torch.int16, device="cuda")[:na]
    ob = torch.empty(max(nb, 1), dtype=torch.int16, device="cuda")[:nb]
    ma, mb = scalar(), scalar()
    ma[0], mb[0] = 3.0e6, 4.0e6   # stale: the call zeroes both first
    dg.dg_convert_f16_amax_pair(dev(xa), dev(xb), oa, ob, f[0:1], ma, mb)
    assert dg.dg_sync_status() == dg.DG_OK
    assert np.array_equal(oa.cpu().numpy().view(np.uint16), oracle.convert_f16(xa, np.float32(0.61)))
    assert np.array_equal(ob.cpu().numpy().view(np.uint16), oracle.convert_f16(xb, np.float32(0.61)))
    assert np.float32(ma[0].item()).view(np.uint32) == np.float32(oracle.amax(xa)).view(np.uint32)
    assert np.float32(mb[0].item()).view(np.uint32) == np.float32(oracle.amax(xb)).view(np.uint32)


def test_convert_with_amax_propagates_nan():
    x = synth.normal_f32(3, (5000,))
    x[4321] = np.nan
    out = torch.empty(5000, dtype=torch.int16, device="cuda")
    am = scalar()
    dg.dg_convert_f16_amax(dev(x), out, None, am)
    assert dg.dg_sync_status() == dg.DG_OK
    assert np.isnan(am[0].item())


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("M,N,K,mma", [(2, 300, 512, None), (9, 1000, 1040, "0"), (129, 520, 1040, None),
                                       (384, 1000, 2048, None)])
def test_recorded_factor_chain(M, N, K, mma, pair):
    """Delayed dynamic-range scaling: each step converts with the factors
    formed from the previous step's maxima, recorded by the conversions
    themselves.  From the second step on (same operands) every factor, FP16
    operand and output matches the oracle's chain of [DG-FP16] §3.3, and the
    factors the step leaves for the next one are the ones it used."""
    A, B = synth.make_inputs("fp8_256", M=M, N=N, K=K)
    A = A.copy()
    A[0, 3] = 9.0e4
    A[M - 1, K - 1] = -7.0e4
    dA, dB = dev(A), dev(B)
    am_a, am_b = scalar(), scalar()
    f = torch.tensor([1.0, 1.0, 1.0, 1.0], dtype=torch.float32, device="cuda")   # no record yet
    A16 = torch.empty((M, K), dtype=torch.int16, device="cuda")
    B16 = torch.empty((N, K), dtype=torch.int16, device="cuda")
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")

    def step():
        if pair:
            dg.dg_convert_f16_amax_pair(dA, dB, A16, B16, f[1:2], am_a, am_b)
        else:
            dg.dg_convert_f16_amax(dA, A16, f[1:2], am_a)
            dg.dg_convert_f16_amax(dB, B16, f[1:2], am_b)
        dg.dg_hgemm_scaled(A16, B16, D, f[2:3], f[3:4], dg.DG_BF16)
        used = f.clone()
        dg.dg_fp16_range_scale(am_a, am_b, f)      # factors for the next step
        return used

    with knobs(DG_MMA_GEMV=mma):
        step()
        used = step()
        assert dg.dg_sync_status() == dg.DG_OK
    fr, A16r, B16r, Dr, S = oracle.fp16_range_chain(A, B)
    assert np.array_equal(used.cpu().numpy().view(np.uint32), fr.view(np.uint32))
    assert np.array_equal(f.cpu().numpy().view(np.uint32), fr.view(np.uint32))
    assert np.array_equal(A16.cpu().numpy().view(np.uint16), A16r)
    assert np.array_equal(B16.cpu().numpy().view(np.uint16), B16r)
    R, _ = oracle.hgemm(A16r, B16r)
    check_bf16_like(bf16_bits_to_f64(D.cpu().numpy().view(np.uint16)), R, S,
                    float(fr[2]), 1.0, "recorded-factor HGEMM")

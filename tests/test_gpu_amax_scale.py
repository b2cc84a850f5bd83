"""The scale formed by the reduction's last CTA (dg_amax, dg_amax_pow2,
dg_quantize_e4m3_amax), against the oracle, bit for bit.

The zeroing kernel also zeroes the scale word, every CTA of the reduction
counts its arrival there after its atomicMax, and the last one writes the
scale over the count.  Covered: one-CTA and many-CTA grids, ragged tails,
back-to-back calls on the same words (the count must start from zero each
time), NaN propagation, the power-of-two scale, and the aliased cases that
keep the separate scale kernel: n == 0, scale_out == amax_out, and the
fused quantiser's next scale written in place over the scale it reads.
"""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def _words(k=3):
    return [torch.full((4,), 123.0, dtype=torch.float32, device="cuda") for _ in range(k)]


def _bits(t):
    return t[0:1].cpu().numpy().view(np.uint32)[0]


def _f32bits(v):
    return np.float32(v).view(np.uint32)


@pytest.mark.parametrize("n", [1, 3, 1000, 131075, 1 << 22, (1 << 24) + 5])
def test_amax_scale_sizes(n):
    x = synth.make_inputs("fp8_8192_e4m3out", M=1, N=1, K=n)[0].reshape(-1)
    xd = torch.from_numpy(x).cuda()
    am, sc, sp = _words()
    dg.dg_amax(xd, am, sc)
    a2, p2 = _words(2)
    dg.dg_amax_pow2(xd, a2, p2)
    assert dg.dg_sync_status() == dg.DG_OK
    ref = oracle.amax(x)
    assert _bits(am) == _f32bits(ref) and _bits(a2) == _f32bits(ref)
    assert _bits(sc) == _f32bits(oracle.scale_from_amax(ref))
    assert _bits(p2) == _f32bits(oracle.scale_pow2_from_amax(ref))


def test_back_to_back_calls_restart_the_count():
    am, sc = _words(2)
    rng = np.random.default_rng(5)
    for i in range(6):
        x = (rng.standard_normal(3_000_001) * (i + 1)).astype(np.float32)
        dg.dg_amax(torch.from_numpy(x).cuda(), am, sc)
        assert dg.dg_sync_status() == dg.DG_OK
        ref = oracle.amax(x)
        assert _bits(am) == _f32bits(ref), i
        assert _bits(sc) == _f32bits(oracle.scale_from_amax(ref)), i


def test_nan_and_zero():
    x = np.zeros(100_000, np.float32)
    am, sc = _words(2)
    dg.dg_amax(torch.from_numpy(x).cuda(), am, sc)
    assert dg.dg_sync_status() == dg.DG_OK
    assert am[0].item() == 0.0 and sc[0].item() == 1.0
    x[77_777] = np.nan
    dg.dg_amax(torch.from_numpy(x).cuda(), am, sc)
    assert dg.dg_sync_status() == dg.DG_OK
    assert np.isnan(am[0].item()) and np.isnan(sc[0].item())


def test_aliased_and_empty_keep_the_scale_kernel():
    x = np.random.default_rng(6).standard_normal(500_000).astype(np.float32)
    ref = oracle.amax(x)
    (w,) = _words(1)
    dg.dg_amax(torch.from_numpy(x).cuda(), w, w)         # scale over amax
    am, sc = _words(2)
    dg.dg_amax(torch.zeros(0, dtype=torch.float32, device="cuda"), am, sc)   # n == 0
    assert dg.dg_sync_status() == dg.DG_OK
    assert _bits(w) == _f32bits(oracle.scale_from_amax(ref))
    assert am[0].item() == 0.0 and sc[0].item() == 1.0


@pytest.mark.parametrize("in_place", [False, True])
def test_fused_quantise_next_scale(in_place):
    A = synth.make_inputs("fp8_sweep_m65", M=300, N=1, K=7777)[0].reshape(-1)
    xd = torch.from_numpy(A).cuda()
    s0 = np.float32(0.01)
    scale = torch.full((4,), float(s0), dtype=torch.float32, device="cuda")
    nxt = scale if in_place else torch.full((4,), 5.0, dtype=torch.float32, device="cuda")
    am = torch.full((4,), 9.0, dtype=torch.float32, device="cuda")
    q = torch.empty(A.shape, dtype=torch.uint8, device="cuda")
    for _ in range(3):   # repeated: the next scale's count restarts every call
        if in_place:
            scale[0] = float(s0)
        dg.dg_quantize_e4m3_amax(xd, scale, q, am, nxt)
        assert dg.dg_sync_status() == dg.DG_OK
        assert np.array_equal(q.cpu().numpy(), oracle.quantize_e4m3(A, s0))
        ref = oracle.amax(A)
        assert _bits(am) == _f32bits(ref)
        assert _bits(nxt) == _f32bits(oracle.scale_from_amax(ref))

"""dg_quantize_e4m3_pair (amax, scale and E4M3 codes of both GEMM operands
in one call) against the oracle and against dg_amax + dg_quantize_e4m3 on
each tensor, bit for bit: sizes with ragged tails in the same or different
CTAs, one empty tensor, an all-zero tensor (scale 1), NaN propagation,
stale words, and repeated calls (the arrival count restarts each time)."""
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


def _w(v=777.0):
    return torch.full((4,), v, dtype=torch.float32, device="cuda")


def _bits(t):
    return t[0:1].cpu().numpy().view(np.uint32)[0]


def _f(v):
    return np.float32(v).view(np.uint32)


def _run(xa, xb):
    da, db = torch.from_numpy(xa).cuda(), torch.from_numpy(xb).cuda()
    qa = torch.empty(max(xa.size, 1), dtype=torch.uint8, device="cuda")[:xa.size]
    qb = torch.empty(max(xb.size, 1), dtype=torch.uint8, device="cuda")[:xb.size]
    ma, mb, sa, sb = _w(), _w(), _w(), _w()
    dg.dg_quantize_e4m3_pair(da, db, ma, mb, sa, sb, qa, qb)
    assert dg.dg_sync_status() == dg.DG_OK
    return ma, mb, sa, sb, qa.cpu().numpy(), qb.cpu().numpy()


def _check(xa, xb, res):
    ma, mb, sa, sb, qa, qb = res
    for x, m, s, q in ((xa, ma, sa, qa), (xb, mb, sb, qb)):
        ref = oracle.amax(x)
        assert _bits(m) == _f(ref)
        sc = oracle.scale_from_amax(ref)
        assert _bits(s) == _f(sc)
        if x.size and not np.isnan(sc):
            assert np.array_equal(q, oracle.quantize_e4m3(x, sc))


@pytest.mark.parametrize("na,nb", [(0, 0), (0, 1000), (777, 0), (100, 77), (4097, (1 << 20) + 7),
                                   ((1 << 22) + 3, (1 << 22) + 5)])
def test_pair_matches_oracle(na, nb):
    xa = synth.normal_f32(90 + na % 7, (na,)) * np.float32(3.0)
    xb = synth.normal_f32(95 + nb % 11, (nb,)) * np.float32(0.02)
    _check(xa, xb, _run(xa, xb))


def test_pair_equals_single_calls():
    A, B = synth.make_inputs("fp8_4096")
    xa, xb = A.reshape(-1)[: (1 << 22) + 9], B.reshape(-1)[: (1 << 21) + 1]
    ma, mb, sa, sb, qa, qb = _run(xa, xb)
    for x, m, s, q in ((xa, ma, sa, qa), (xb, mb, sb, qb)):
        d = torch.from_numpy(x).cuda()
        am, sc = _w(), _w()
        q1 = torch.empty(x.size, dtype=torch.uint8, device="cuda")
        dg.dg_amax(d, am, sc)
        dg.dg_quantize_e4m3(d, sc, q1)
        assert dg.dg_sync_status() == dg.DG_OK
        assert _bits(am) == _bits(m) and _bits(sc) == _bits(s)
        assert np.array_equal(q1.cpu().numpy(), q)


def test_zero_and_nan():
    xa = np.zeros(10_000, np.float32)
    xb = synth.normal_f32(5, (20_000,))
    xb[12_345] = np.nan
    ma, mb, sa, sb, qa, qb = _run(xa, xb)
    assert ma[0].item() == 0.0 and sa[0].item() == 1.0 and not qa.any()
    assert np.isnan(mb[0].item()) and np.isnan(sb[0].item())


def test_repeated_calls_restart_the_count():
    rng = np.random.default_rng(3)
    da = torch.empty(2_000_003, dtype=torch.float32, device="cuda")
    db = torch.empty(1_000_001, dtype=torch.float32, device="cuda")
    qa = torch.empty(da.numel(), dtype=torch.uint8, device="cuda")
    qb = torch.empty(db.numel(), dtype=torch.uint8, device="cuda")
    ma, mb, sa, sb = _w(), _w(), _w(), _w()
    for i in range(5):
        xa = (rng.standard_normal(da.numel()) * (i + 1)).astype(np.float32)
        xb = (rng.standard_normal(db.numel()) * (5 - i)).astype(np.float32)
        da.copy_(torch.from_numpy(xa))
        db.copy_(torch.from_numpy(xb))
        dg.dg_quantize_e4m3_pair(da, db, ma, mb, sa, sb, qa, qb)
        assert dg.dg_sync_status() == dg.DG_OK
        _check(xa, xb, (ma, mb, sa, sb, qa.cpu().numpy(), qb.cpu().numpy()))

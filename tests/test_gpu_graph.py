"""The whole path (amax, scale, quantise, GEMM) captured into a CUDA graph and
replayed gives bit-identical results to direct calls, on each kernel path."""
import numpy as np
import pytest
import torch

import fp16_tensor_core_gb300 as dg
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp16_tensor_core_gb300 import build
    build.build()
    dg.dg_init()   # per-device set-up happens before any capture
    yield
    assert dg.dg_sync_status() == dg.DG_OK


def chain(A, B, bufs, out):
    qa, qb, sa, sb, am_a, am_b, sd, D = bufs
    dg.dg_amax(A, am_a, sa)
    dg.dg_amax(B, am_b, sb)
    dg.dg_quantize_e4m3(A, sa, qa)
    dg.dg_quantize_e4m3(B, sb, qb)
    dg.dg_fp8_gemm(qa, qb, D, sa, sb, sd, out)


@pytest.mark.parametrize("M,N,K,out", [
    (1, 1000, 1040, dg.DG_BF16),      # warp-MMA GEMV
    (16, 4096, 1040, dg.DG_BF16),     # split-K (32 tiles, each over four CTAs)
    (129, 1000, 1040, dg.DG_BF16),    # single CTA
    (640, 1536, 2048, dg.DG_E4M3),    # CTA pairs, E4M3 out
])
def test_graph_replay_matches_direct_calls(M, N, K, out):
    A32, B32 = synth.make_inputs("fp8_sweep_m65", M=M, N=N, K=K)
    A, B = torch.from_numpy(A32).cuda(), torch.from_numpy(B32).cuda()
    f = lambda: torch.zeros(4, dtype=torch.float32, device="cuda")  # noqa: E731
    sd = f()
    sd[0] = 2.0
    dt = torch.uint8 if out == dg.DG_E4M3 else torch.int16

    def bufs():
        return (torch.empty((M, K), dtype=torch.uint8, device="cuda"),
                torch.empty((N, K), dtype=torch.uint8, device="cuda"), f(), f(), f(), f(), sd,
                torch.empty((M, N), dtype=dt, device="cuda"))

    direct = bufs()
    chain(A, B, direct, out)
    assert dg.dg_sync_status() == dg.DG_OK

    captured = bufs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain(A, B, captured, out)          # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    captured[-1].zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain(A, B, captured, out)
    for _ in range(2):
        captured[-1].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert dg.dg_sync_status() == dg.DG_OK
        for a, b in zip(direct, captured):
            assert torch.equal(a, b)

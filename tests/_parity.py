"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI and compare it with the CPU oracle under the stated tolerances.

Tolerances ([FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南"):
* amax, scale, E4M3 codes of the quantiser: bit-exact.
* BF16 / FP16 GEMM output: |D - Dref| <= 8e-3 |Dref| + 1e-4 S sA sB per
  element, Dref = sA sB sum_k a b in FP64 and S = sum_k |a b|.
* E4M3 GEMM output: at most 1 E4M3 step from e4m3(Dref / sD) in the
  ordered code space (+0 and -0 are the same point).
"""
from __future__ import annotations

import numpy as np
import torch

import fp16_tensor_core_gb300 as dg
import oracle

REL, ABS = 8e-3, 1e-4


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def scalar() -> torch.Tensor:
    return torch.zeros(4, dtype=torch.float32, device="cuda")  # 16 B, own allocation


def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def fp16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return u16.view(np.float16).astype(np.float64)


def ordered(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def gpu_quantize(x32: np.ndarray):
    """Device amax -> scale -> quantise of one FP32 tensor (via the C ABI)."""
    dx = dev(x32)
    amax, scale = scalar(), scalar()
    dg.dg_amax(dx, amax, scale)
    q = torch.empty(dx.shape, dtype=torch.uint8, device="cuda")
    dg.dg_quantize_e4m3(dx, scale, q)
    return q, amax, scale


def check_quantised(x32, q_dev, amax_dev, scale_dev):
    """Bit-exact comparison of one tensor's device quantisation with the oracle."""
    q_ref, s_ref, a_ref = oracle.quantize_tensor(x32)
    a = amax_dev[0:1].cpu().numpy()
    s = scale_dev[0:1].cpu().numpy()
    assert a.view(np.uint32)[0] == np.float32(a_ref).view(np.uint32), (a, a_ref)
    assert s.view(np.uint32)[0] == np.float32(s_ref).view(np.uint32), (s, s_ref)
    q = q_dev.cpu().numpy()
    bad = np.flatnonzero(q.reshape(-1) != q_ref.reshape(-1))
    assert bad.size == 0, f"{bad.size} codes differ, first at {bad[:5]}: " \
        f"gpu {q.reshape(-1)[bad[:5]]} oracle {q_ref.reshape(-1)[bad[:5]]} x {x32.reshape(-1)[bad[:5]]}"
    return q_ref, np.float32(s_ref)


def check_bf16_like(d_f64, R, S, sa, sb, what="BF16"):
    dref = oracle.epilogue_scale(R, sa, sb)
    bound = REL * np.abs(dref) + ABS * S * float(sa) * float(sb)
    err = np.abs(d_f64 - dref)
    bad = np.flatnonzero(~(err <= bound))
    assert bad.size == 0, (f"{what}: {bad.size}/{err.size} outside tolerance; first {bad[:5]} "
                           f"got {d_f64.reshape(-1)[bad[:5]]} want {dref.reshape(-1)[bad[:5]]} "
                           f"bound {bound.reshape(-1)[bad[:5]]}")
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


def check_e4m3(codes, R, sa, sb, sd):
    ref = oracle.epilogue_e4m3(R, sa, sb, sd)
    dist = np.abs(ordered(codes) - ordered(ref))
    bad = np.flatnonzero(dist > 1)
    assert bad.size == 0, (f"E4M3 out: {bad.size} codes more than 1 step away; first {bad[:5]} "
                           f"gpu {codes.reshape(-1)[bad[:5]]} oracle {ref.reshape(-1)[bad[:5]]}")
    return int(dist.max()) if dist.size else 0


def sample_positions(M, N, count, seed=1, tile_m=128, tile_n=64):
    """Seeded random (m, n) plus corners and tile-boundary rows/columns."""
    rng = np.random.default_rng(seed)
    ms = list(rng.integers(0, M, count))
    ns = list(rng.integers(0, N, count))
    edge_m = sorted({0, M - 1, *[min(M - 1, k * tile_m + d) for k in range(1, 4) for d in (-1, 0)]})
    edge_n = sorted({0, N - 1, *[min(N - 1, k * tile_n + d) for k in range(1, 4) for d in (-1, 0)]})
    for m in edge_m:
        for n in edge_n:
            ms.append(m)
            ns.append(n)
    return np.array(ms, dtype=np.int64), np.array(ns, dtype=np.int64)


def guarded(numel: int, dtype: torch.dtype, sentinel: int, guard: int = 64):
    """A device buffer with `guard` sentinel elements on each side of the
    output region; returns (whole buffer, output view)."""
    buf = torch.full((numel + 2 * guard,), sentinel, dtype=dtype, device="cuda")
    return buf, buf[guard:guard + numel]


def check_guards(buf: torch.Tensor, numel: int, sentinel: int, guard: int = 64):
    h = buf.cpu().numpy()
    assert np.all(h[:guard] == sentinel) and np.all(h[guard + numel:] == sentinel), \
        "write outside [0, M) x [0, N)"

"""Seeded synthetic inputs shared by the tests, the oracle scripts and the bench.

This module holds no GEMM or quantiser arithmetic: it only draws the FP32 /
FP16 input matrices that the pages' workloads describe, and it draws them the
same way on every machine.  The pages give no dataset; every workload is
random matrices of the stated shapes and distributions:

* [FP8-guide] "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南" §4.3 (random
  matrices checked against an FP32 product), §3.3 (edge sizes 1, 63, 65, 127,
  129), §2.2 (a 4096^3 FP8 GEMM), §5.4 (all-ones matrices).
* the DeepGEMM FP16/WMMA deep-dive page §2.1 and §4.1: the decode QKV
  projection [1, 4096] x [4096, 12288].
* "HGEMM优化：深度学习中的矩阵乘法性能提升策略" §4: FP16 square GEMMs.

Random numbers come from a counter-based generator: value i of stream `seed`
is SplitMix64 (Steele, Lea and Flood, OOPSLA 2014; the constants of Vigna's
reference `splitmix64.c`) applied to `seed * 2^32 + i`.  Normals use the
Marsaglia-Bray polar method; its logarithm is computed here with basic IEEE
operations only (frexp plus an atanh series), so no libm or SIMD math library
can change a bit between x86-64 and AArch64.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_LN2 = 0.6931471805599453094
_CHUNK = 1 << 22


def _splitmix64(counter: np.ndarray) -> np.ndarray:
    """SplitMix64 output for the given 64-bit counters (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = counter * _GAMMA + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform(seed: int, start: int, count: int) -> np.ndarray:
    """Doubles in [0, 1): the top 53 bits of draws start .. start+count-1."""
    base = np.uint64((seed & 0xFFFFFFFF) << 32)
    idx = np.arange(start, start + count, dtype=np.uint64) + base
    return (_splitmix64(idx) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _ln(x: np.ndarray) -> np.ndarray:
    """Natural log of positive finite doubles from +, -, *, / and frexp only."""
    m, e = np.frexp(x)                      # x = m * 2^e, m in [0.5, 1)
    small = m < 0.7071067811865476
    m = np.where(small, m * 2.0, m)
    e = np.where(small, e - 1, e).astype(np.float64)
    t = (m - 1.0) / (m + 1.0)               # |t| < 0.1716
    t2 = t * t
    acc = np.full_like(t, 1.0 / 23.0)
    for d in (21.0, 19.0, 17.0, 15.0, 13.0, 11.0, 9.0, 7.0, 5.0, 3.0, 1.0):
        acc = acc * t2 + 1.0 / d
    return e * _LN2 + 2.0 * t * acc


def normal(seed: int, count: int, start_pair: int = 0) -> np.ndarray:
    """`count` N(0,1) doubles by the polar method over pairs of draws."""
    out = np.empty(count, dtype=np.float64)
    filled = 0
    pair = start_pair
    while filled < count:
        want = count - filled
        npairs = max(1024, min(_CHUNK, int(want * 0.66) + 1024))
        u = uniform(seed, 2 * pair, 2 * npairs).reshape(npairs, 2)
        pair += npairs
        v = 2.0 * u - 1.0
        s = v[:, 0] * v[:, 0] + v[:, 1] * v[:, 1]
        ok = (s > 0.0) & (s < 1.0)
        v = v[ok]
        s = s[ok]
        f = np.sqrt(-2.0 * _ln(s) / s)
        z = (v * f[:, None]).reshape(-1)
        take = min(z.size, want)
        out[filled:filled + take] = z[:take]
        filled += take
    return out


def normal_f32(seed: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    z = normal(seed, n)
    if std != 1.0:
        z = z * std
    return z.astype(np.float32).reshape(shape)


def uniform_f32(seed: int, shape, lo: float, hi: float, start: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    u = uniform(seed, start, n)
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def random_bytes(seed: int, shape, start: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    base = np.uint64((seed & 0xFFFFFFFF) << 32)
    idx = np.arange(start, start + n, dtype=np.uint64) + base
    return (_splitmix64(idx) >> np.uint64(56)).astype(np.uint8).reshape(shape)


# -- the workloads ------------------------------------------------------------

#: name -> (M, N, K, kind).  kind: "fp8" (E4M3 GEMM, BF16 out), "fp8_e4m3out",
#: "fp16" (HGEMM, FP16 out).
CONFIGS = {
    "fp8_256": (256, 256, 256, "fp8"),
    "fp8_sweep_m1": (1, 1000, 1040, "fp8"),
    "fp8_sweep_m63": (63, 1000, 1040, "fp8"),
    "fp8_sweep_m65": (65, 1000, 1040, "fp8"),
    "fp8_sweep_m129": (129, 1000, 1040, "fp8"),
    "fp8_qkv": (1, 12288, 4096, "fp8"),
    "fp8_4096": (4096, 4096, 4096, "fp8"),
    "fp16_4096": (4096, 4096, 4096, "fp16"),
    "fp8_8192_e4m3out": (8192, 8192, 8192, "fp8_e4m3out"),
}


def make_inputs(name: str, M: int | None = None, N: int | None = None,
                K: int | None = None):
    """FP32 (or FP16 bit patterns, for "fp16") A (M x K) and B (N x K).

    Shapes default to the named workload; overriding them keeps its
    distribution (used for reduced-size parity cases).

    * all streams: seed 0, A drawn first (row-major), then B.
    * fp8_sweep_*: additionally each entry, independently with probability
      0.001 (stream seed 1, same A-then-B order), is multiplied by 50.
    * fp8_qkv: A ~ N(0, 1), B ~ N(0, 0.02^2).
    * fp16_4096: U(-1, 1) in FP32, then round-to-nearest-even to FP16.
    * everything else: N(0, 1).
    """
    M0, N0, K0, kind = CONFIGS[name]
    M = M0 if M is None else M
    N = N0 if N is None else N
    K = K0 if K is None else K
    na, nb = M * K, N * K
    if kind == "fp16":
        u = uniform(0, 0, na + nb)
        x = (-1.0 + 2.0 * u).astype(np.float32).astype(np.float16)
        A = x[:na].view(np.uint16).reshape(M, K).copy()
        B = x[na:].view(np.uint16).reshape(N, K).copy()
        return A, B
    z = normal(0, na + nb)
    if name == "fp8_qkv":
        z[na:] *= 0.02
    if name.startswith("fp8_sweep"):
        hit = uniform(1, 0, na + nb) < 0.001
        z[hit] *= 50.0
    x = z.astype(np.float32)
    return x[:na].reshape(M, K).copy(), x[na:].reshape(N, K).copy()


def moe_group_sizes(seed: int, groups: int, total: int, empty: int = 0) -> np.ndarray:
    """Skewed expert loads summing to `total` (a mixture-of-experts routing
    mix): weights u^3 + 0.02 from the counter stream, floor-rounded, the
    remainder spread one row at a time over the largest groups; the first
    `empty` groups get no rows."""
    u = uniform(seed, 0, groups)
    w = u * u * u + 0.02
    w[:empty] = 0.0
    sizes = np.floor(total * w / w.sum()).astype(np.int64)
    rest = total - int(sizes.sum())
    order = np.argsort(-w, kind="stable")
    for i in range(rest):
        sizes[order[i % (groups - empty)]] += 1
    return sizes


def make_moe_inputs(groups: int, total: int, N: int, K: int, seed: int = 0, empty: int = 0):
    """FP32 A (total x K, groups' rows stacked), FP32 B (groups*N x K) and
    int32 offsets [groups + 1]; A and B ~ N(0, 1) from stream `seed`, A first."""
    sizes = moe_group_sizes(seed + 7, groups, total, empty)
    offs = np.zeros(groups + 1, dtype=np.int32)
    offs[1:] = np.cumsum(sizes)
    z = normal(seed, total * K + groups * N * K).astype(np.float32)
    return (z[:total * K].reshape(total, K).copy(), z[total * K:].reshape(groups * N, K).copy(),
            offs)

"""Benchmark: the per-tensor-scaled E4M3 GEMM path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch of synthetic input,
the 8192 x 8192 x 8192 E4M3 workload with E4M3 output:
    amax(A), amax(B) -> scale = amax/448 -> quantise(A), quantise(B)
    -> tensor-core GEMM, D = E4M3(sA*sB*(A_q @ B_q^T) / sD)
with FP32 A and B resident in HBM (2 x 268 MB, larger than the 129 MB L2).
`value` is whole-step throughput in TFLOPS (2*M*N*K per step); `roofline`
rates the dominant kernel (the GEMM) on its own CUDA-event launch time;
`e2e` repeats the step through the public API with the FP32 inputs copied
from pinned host memory and D copied back inside the timed region; `extra`
lists kernel-level numbers for the other workloads (decode QKV GEMV GB/s,
4096^3 FP8 and FP16 TFLOPS, amax/quantise GB/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl own|reference]

`--impl reference` times the CPU oracle (the only reference this method has)
on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M = N = K = 8192
FLOP_PER_STEP = 2.0 * M * N * K
WORKLOAD = "fp8_8192_e4m3out"
CPU_SAMPLE_ROWS = 3072  # ~10-20 s of oracle work on 16 cores
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
# Nominal dense FP8 tensor rate of one GB300 (NVIDIA's figure without 2:4
# sparsity), for context beside the measured-peak fraction.
NOMINAL_FP8_TFLOPS = 4500.0


# ---------------------------------------------------------------- plumbing

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-workload kernel numbers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", default=None, help="time one kernel workload alone")
    ap.add_argument("--graph", action="store_true",
                    help="with --kernel: also time the launches replayed from a CUDA graph")
    ap.add_argument("--record-traffic", nargs="+", default=None, metavar="WORKLOAD=CSV",
                    help="write profiles/traffic.json from ncu CSV logs (no GPU work)")
    ap.add_argument("--settle-seconds", type=float, default=1.5,
                    help="untimed busy period before the timed steps (clock sampling)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def source_hash(files) -> str:
    """First 16 hex digits of the SHA-256 of the named kernel sources."""
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "fp16_tensor_core_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of `workload`'s kernel from the committed ncu
    summary, if it was taken on the kernel's current sources; else None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    for e in rec.get("entries", []):
        if e.get("workload") == workload and e.get("source_sha256_16") == source_hash(e["sources"]):
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                             "hw": parts[5], "hwth": parts[6], "swth": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        pmax = max(r["power"] for r in rows)
        load = [r for r in rows if r["power"] >= 0.5 * pmax] or rows
        reasons = set()
        for r in load:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwth"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swth"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": pmax}


# ------------------------------------------------------------ own workload

GEMM_EVENT_EVERY = 5   # timed steps that carry the GEMM's event pair: 0, 5, 10, ...


class Workload:
    """Device buffers for one step of the 8192^3 E4M3-output path."""

    def __init__(self, torch, dg, A32, B32, sd: float):
        self.torch, self.dg = torch, dg
        dev = "cuda"
        self.A = torch.from_numpy(A32).to(dev)
        self.B = torch.from_numpy(B32).to(dev)
        f = lambda: torch.zeros(4, dtype=torch.float32, device=dev)  # noqa: E731
        self.amax_a, self.amax_b, self.sa, self.sb, self.sd = f(), f(), f(), f(), f()
        self.sd[0] = sd
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        self.qb = torch.empty((N, K), dtype=torch.uint8, device=dev)
        self.D = torch.empty((M, N), dtype=torch.uint8, device=dev)

    def step(self, stream, ev=None):
        dg = self.dg
        # amax and scale of A and B, then both quantised (one call, three
        # launches: bit-identical to dg_amax + dg_quantize_e4m3 on each)
        dg.dg_quantize_e4m3_pair(self.A, self.B, self.amax_a, self.amax_b, self.sa, self.sb,
                                 self.qa, self.qb, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        dg.dg_fp8_gemm(self.qa, self.qb, self.D, self.sa, self.sb, self.sd, dg.DG_E4M3,
                       stream=stream)
        if ev is not None:
            ev[1].record(stream)

    KERNELS_PER_STEP = 4  # zeroing, amax of A and B (with scales), quantise of A and B, GEMM


def time_kernel(torch, stream, fn, iters: int, warmup: int = 3) -> float:
    """Mean milliseconds per call of fn(i) measured with CUDA events."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(iters):
        fn(i)
    e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) / iters


def time_graph(torch, fn, iters: int, warmup: int = 3, reps: int = 5) -> float:
    """Mean milliseconds per call of fn(i, stream) when the `iters` calls are
    captured once into a CUDA graph and the graph is replayed: the device
    time of back-to-back launches without the per-call host cost."""
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        for i in range(warmup):
            fn(i, cap)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for i in range(iters):
            fn(i, cap)
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(cur)
    for _ in range(reps):
        g.replay()
    e.record(cur)
    e.synchronize()
    return s.elapsed_time(e) / (reps * iters)


def kernel_cases(torch, dg):
    """Single-kernel workloads for the `extra` numbers, `--kernel` runs and
    ncu captures.  Operands that would stay L2-resident between launches are
    rotated over several copies (together more than 3 x L2)."""
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    dev = "cuda"

    def codes(shape, seed):
        # timing only: any E4M3 code pattern (NaN codes avoided)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        t = torch.randint(0, 256, shape, dtype=torch.uint8, device=dev, generator=g)
        return torch.where((t & 0x7F) == 0x7F, torch.zeros_like(t), t)

    def ncopies(nbytes):
        return max(1, int(3 * l2 // max(nbytes, 1)) + 1)

    one = torch.ones(4, dtype=torch.float32, device=dev)

    def qkv():
        Mq, Nq, Kq = 1, 12288, 4096
        nb = ncopies(Nq * Kq)
        As = [codes((Mq, Kq), 10 + i) for i in range(nb)]
        Bs = [codes((Nq, Kq), 20 + i) for i in range(nb)]
        D = torch.empty((Mq, Nq), dtype=torch.bfloat16, device=dev)
        fn = lambda i, s: dg.dg_fp8_gemm(As[i % nb], Bs[i % nb], D, one, one, None,  # noqa: E731
                                         dg.DG_BF16, stream=s)
        return fn, 2.0 * Mq * Nq * Kq, Nq * Kq + Mq * Kq + Mq * Nq * 2, "hbm", f"{nb} rotating copies"

    def gemv_m(m, Nq=12288, Kq=4096):
        nb = ncopies(Nq * Kq)
        As = [codes((m, Kq), 70 + i) for i in range(nb)]
        Bs = [codes((Nq, Kq), 80 + i) for i in range(nb)]
        D = torch.empty((m, Nq), dtype=torch.bfloat16, device=dev)
        fn = lambda i, s: dg.dg_fp8_gemm(As[i % nb], Bs[i % nb], D, one, one, None,  # noqa: E731
                                         dg.DG_BF16, stream=s)
        return fn, 2.0 * m * Nq * Kq, Nq * Kq + m * Kq + m * Nq * 2, "hbm", f"{nb} rotating copies"

    def small_fp8(M, N, K):
        # latency-bound parity configurations (256^3, the 1000 x 1040 sweep)
        nb = ncopies(M * K + N * K)
        As = [codes((M, K), 90 + i) for i in range(nb)]
        Bs = [codes((N, K), 95 + i) for i in range(nb)]
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda i, s: dg.dg_fp8_gemm(As[i % nb], Bs[i % nb], D, one, one, None,  # noqa: E731
                                         dg.DG_BF16, stream=s)
        return fn, 2.0 * M * N * K, M * K + N * K + 2 * M * N, "latency", f"{nb} rotating copies"

    def fp8_sq(S, out):
        nb = ncopies(2 * S * S)
        As = [codes((S, S), 30 + i) for i in range(nb)]
        Bs = [codes((S, S), 40 + i) for i in range(nb)]
        D = torch.empty((S, S), dtype=torch.uint8 if out == dg.DG_E4M3 else torch.bfloat16, device=dev)
        fn = lambda i, s: dg.dg_fp8_gemm(As[i % nb], Bs[i % nb], D, one, one, one, out,  # noqa: E731
                                         stream=s)
        return fn, 2.0 * S ** 3, 2 * S * S + S * S * (1 if out == dg.DG_E4M3 else 2), "tensor_fp8", \
            f"{nb} rotating copies"

    def hgemm(S):
        nb = ncopies(4 * S * S)
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        Hs = [(torch.rand((S, S), device=dev, generator=g) * 2 - 1).half() for _ in range(nb)]
        Hb = [(torch.rand((S, S), device=dev, generator=g) * 2 - 1).half() for _ in range(nb)]
        D = torch.empty((S, S), dtype=torch.float16, device=dev)
        fn = lambda i, s: dg.dg_hgemm(Hs[i % nb], Hb[i % nb], D, dg.DG_FP16, stream=s)  # noqa: E731
        return fn, 2.0 * S ** 3, 6 * S * S, "tensor_fp16", f"{nb} rotating copies"

    def hgemv(m, Nq=12288, Kq=4096):
        # FP16 operands on the decode QKV shape (the HGEMM's GEMV path)
        nb = ncopies(2 * Nq * Kq)
        g = torch.Generator(device=dev)
        g.manual_seed(6)
        Ha = [(torch.rand((m, Kq), device=dev, generator=g) * 2 - 1).half() for _ in range(nb)]
        Hb = [((torch.rand((Nq, Kq), device=dev, generator=g) * 2 - 1) * 0.02).half() for _ in range(nb)]
        D = torch.empty((m, Nq), dtype=torch.float16, device=dev)
        fn = lambda i, s: dg.dg_hgemm(Ha[i % nb], Hb[i % nb], D, dg.DG_FP16, stream=s)  # noqa: E731
        return fn, 2.0 * m * Nq * Kq, 2 * (Nq * Kq + m * Kq + m * Nq), "hbm", f"{nb} rotating copies"

    def amax():
        x = torch.randn((8192, 8192), device=dev)
        am = torch.zeros(4, dtype=torch.float32, device=dev)
        sc = torch.zeros(4, dtype=torch.float32, device=dev)
        fn = lambda i, s: dg.dg_amax(x, am, sc, stream=s)  # noqa: E731
        return fn, 0.0, 4 * x.numel(), "hbm", "268 MB input > L2"

    def quant():
        x = torch.randn((8192, 8192), device=dev)
        sc = torch.full((4,), 0.01, dtype=torch.float32, device=dev)
        q = torch.empty((8192, 8192), dtype=torch.uint8, device=dev)
        fn = lambda i, s: dg.dg_quantize_e4m3(x, sc, q, stream=s)  # noqa: E731
        return fn, 0.0, 5 * x.numel(), "hbm", "268 MB input > L2"

    def quant_amax():
        x = torch.randn((8192, 8192), device=dev)
        sc = torch.full((4,), 0.01, dtype=torch.float32, device=dev)
        am = torch.zeros(4, dtype=torch.float32, device=dev)
        nx = torch.zeros(4, dtype=torch.float32, device=dev)
        q = torch.empty((8192, 8192), dtype=torch.uint8, device=dev)
        fn = lambda i, s: dg.dg_quantize_e4m3_amax(x, sc, q, am, nx, stream=s)  # noqa: E731
        return fn, 0.0, 5 * x.numel(), "hbm", "268 MB input > L2"

    def convert16():
        x = torch.randn((8192, 8192), device=dev)
        f = torch.full((4,), 0.25, dtype=torch.float32, device=dev)
        o = torch.empty((8192, 8192), dtype=torch.int16, device=dev)
        fn = lambda i, s: dg.dg_convert_f16(x, o, f, stream=s)  # noqa: E731
        return fn, 0.0, 6 * x.numel(), "hbm", "268 MB input > L2"

    def fp16_range_chain(S):
        # FP32 operands with values beyond FP16 range: amax of both, the
        # dynamic-range factors, sqrt(scale) conversion of both, scaled HGEMM
        g = torch.Generator(device=dev)
        g.manual_seed(9)
        A = torch.randn((S, S), device=dev, generator=g)
        B = torch.randn((S, S), device=dev, generator=g)
        A[0, 0] = 9.0e4
        am_a, am_b, f = (torch.zeros(4, dtype=torch.float32, device=dev) for _ in range(3))
        A16 = torch.empty((S, S), dtype=torch.int16, device=dev)
        B16 = torch.empty((S, S), dtype=torch.int16, device=dev)
        D = torch.empty((S, S), dtype=torch.bfloat16, device=dev)

        def fn(i, s):
            dg.dg_amax(A, am_a, stream=s)
            dg.dg_amax(B, am_b, stream=s)
            dg.dg_fp16_range_scale(am_a, am_b, f, stream=s)
            dg.dg_convert_f16(A, A16, f[1:2], stream=s)
            dg.dg_convert_f16(B, B16, f[1:2], stream=s)
            dg.dg_hgemm_scaled(A16, B16, D, f[2:3], f[3:4], dg.DG_BF16, stream=s)
        return fn, 2.0 * S ** 3, 0.0, "tensor_fp16", "FP32 operands 2 x 67 MB (> L2 together with the FP16 copies)"

    def fp16_range_recorded_chain(S):
        # the same chain with delayed scaling: each step converts with the
        # factors of the previous step's maxima, recorded by the conversions
        # (one read of each FP32 operand instead of two), then forms the next
        # factors
        g = torch.Generator(device=dev)
        g.manual_seed(9)
        A = torch.randn((S, S), device=dev, generator=g)
        B = torch.randn((S, S), device=dev, generator=g)
        A[0, 0] = 9.0e4
        am_a, am_b = (torch.zeros(4, dtype=torch.float32, device=dev) for _ in range(2))
        f = torch.ones(4, dtype=torch.float32, device=dev)
        A16 = torch.empty((S, S), dtype=torch.int16, device=dev)
        B16 = torch.empty((S, S), dtype=torch.int16, device=dev)
        D = torch.empty((S, S), dtype=torch.bfloat16, device=dev)

        def fn(i, s):
            # both operands converted (and their maxima recorded) in one pass
            dg.dg_convert_f16_amax_pair(A, B, A16, B16, f[1:2], am_a, am_b, stream=s)
            dg.dg_hgemm_scaled(A16, B16, D, f[2:3], f[3:4], dg.DG_BF16, stream=s)
            dg.dg_fp16_range_scale(am_a, am_b, f, stream=s)
        return fn, 2.0 * S ** 3, 0.0, "tensor_fp16", "FP32 operands 2 x 67 MB (> L2 together with the FP16 copies)"

    def moe(grouped: bool):
        # 16 experts, 8192 routed rows with a skewed load, N = 2048, K = 4096
        import synth
        G, total, Nm, Km = 16, 8192, 2048, 4096
        sizes = synth.moe_group_sizes(7, G, total)
        offs = torch.zeros(G + 1, dtype=torch.int32)
        offs[1:] = torch.from_numpy(sizes.cumsum()).to(torch.int32)
        doffs = offs.to(dev)
        nb = ncopies(total * Km + G * Nm * Km)
        As = [codes((total, Km), 50 + i) for i in range(nb)]
        Bs = [codes((G * Nm, Km), 60 + i) for i in range(nb)]
        sg = torch.ones(G, dtype=torch.float32, device=dev)
        D = torch.empty((total, Nm), dtype=torch.bfloat16, device=dev)
        o = offs.tolist()

        def fn(i, s):
            A, B = As[i % nb], Bs[i % nb]
            if grouped:
                dg.dg_fp8_gemm_grouped(A, B, D, doffs, sg, sg, None, dg.DG_BF16, stream=s,
                                       M=total, N=Nm, K=Km, groups=G)
            else:
                for g in range(G):
                    if o[g + 1] > o[g]:
                        dg.dg_fp8_gemm(A[o[g]:o[g + 1]], B[g * Nm:(g + 1) * Nm], D[o[g]:o[g + 1]],
                                       sg[g:g + 1], sg[g:g + 1], None, dg.DG_BF16, stream=s)
        return fn, 2.0 * total * Nm * Km, total * Km + G * Nm * Km + total * Nm * 2, "tensor_fp8", \
            f"{nb} rotating copies; group sizes {sizes.min()}..{sizes.max()}"

    return {
        "moe_grouped_16x8192x2048x4096": lambda: moe(True),
        "moe_per_group_calls_16x8192x2048x4096": lambda: moe(False),
        "fp8_gemm_256": lambda: small_fp8(256, 256, 256),
        "fp8_sweep_m1_1x1000x1040": lambda: small_fp8(1, 1000, 1040),
        "fp8_sweep_m63_63x1000x1040": lambda: small_fp8(63, 1000, 1040),
        "fp8_sweep_m65_65x1000x1040": lambda: small_fp8(65, 1000, 1040),
        "fp8_sweep_m129_129x1000x1040": lambda: small_fp8(129, 1000, 1040),
        "qkv_gemv_1x12288x4096": qkv,
        "qkv_m4_4x12288x4096": lambda: gemv_m(4),
        "qkv_m8_8x12288x4096": lambda: gemv_m(8),
        "qkv_m16_16x12288x4096": lambda: gemv_m(16),
        "qkv_m32_32x12288x4096": lambda: gemv_m(32),
        "qkv_m64_64x12288x4096": lambda: gemv_m(64),
        "qkv_m128_128x12288x4096": lambda: gemv_m(128),
        "qkv_m256_256x12288x4096": lambda: gemv_m(256),
        # a decode-batch FFN down projection (long K): split-K up to M = 64
        "ffn_down_m16_16x4096x11008": lambda: gemv_m(16, 4096, 11008),
        "ffn_down_m64_64x4096x11008": lambda: gemv_m(64, 4096, 11008),
        "ffn_down_m128_128x4096x11008": lambda: gemv_m(128, 4096, 11008),
        "fp8_gemm_4096": lambda: fp8_sq(4096, dg.DG_BF16),
        "fp8_gemm_8192_e4m3out": lambda: fp8_sq(8192, dg.DG_E4M3),
        "fp16_hgemm_4096": lambda: hgemm(4096),
        "fp16_qkv_gemv_1x12288x4096": lambda: hgemv(1),
        "amax_8192sq": amax,
        "quantise_8192sq": quant,
        "quantise_with_amax_8192sq": quant_amax,
        "convert_f16_8192sq": convert16,
        "fp16_range_scaled_hgemm_chain_4096": lambda: fp16_range_chain(4096),
        "fp16_range_recorded_chain_4096": lambda: fp16_range_recorded_chain(4096),
    }


def measure_case(torch, dg, make, stream, peaks, iters, warmup=3, graph=True) -> dict:
    """Time one kernel workload.  With `graph`, the headline `us` is the
    graph-replayed time (device-bound) and `us_stream` the same calls
    launched one by one from Python (bounded by the host for short kernels)."""
    fn, flop, nbytes, bound, note = make()
    ms_stream = time_kernel(torch, stream, lambda i: fn(i, stream), iters, warmup)
    ms = time_graph(torch, fn, iters, warmup) if graph else ms_stream
    st = dg.dg_sync_status()
    assert st == dg.DG_OK, dg.dg_status_string(st)
    rec = {"us": ms * 1e3, "launch": "graph" if graph else "stream", "GB/s": nbytes / (ms * 1e-3) / 1e9,
           "l2": note}
    if graph:
        rec["us_stream"] = ms_stream * 1e3
    if flop:
        rec["TFLOPS"] = flop / (ms * 1e-3) / 1e12
    if bound == "hbm":
        rec["frac_hbm"] = rec["GB/s"] / peaks["hbm_gbs"]
    elif bound == "tensor_fp8":
        rec["frac_fp8_peak"] = rec["TFLOPS"] / (2.0 * peaks["bf16_tflops"])
    elif bound == "tensor_fp16":
        rec["frac_fp16_peak"] = rec["TFLOPS"] / peaks["bf16_tflops"]
    return rec


def extras(torch, dg, stream, peaks) -> dict:
    out = {}
    for name, make in kernel_cases(torch, dg).items():
        if name == "fp8_gemm_8192_e4m3out":
            continue  # the headline step already times this kernel
        out[name] = measure_case(torch, dg, make, stream, peaks, 50)
        torch.cuda.empty_cache()
    return out


def compact(rec: dict) -> dict:
    """The per-workload numbers that matter, rounded (keeps the line short)."""
    keep = {"us": 2, "us_stream": 2, "TFLOPS": 1, "GB/s": 0, "frac_hbm": 3, "frac_fp8_peak": 3,
            "frac_fp16_peak": 3}
    return {k: round(rec[k], d) for k, d in keep.items() if k in rec}


# The bandwidth-bound decode shapes (the M <= 16 half of the metric): the
# QKV projection weights B[12288, 4096] with M = 1, 8 and 16 rows of A.
SKINNY_ROOFLINES = {"m1": "qkv_gemv_1x12288x4096", "m8": "qkv_m8_8x12288x4096",
                    "m16": "qkv_m16_16x12288x4096"}
KERNEL_OF_PATH = {2: "gemv_kernel (CUDA-core GEMV)", 3: "gemm_tc_kernel (tiled tcgen05)",
                  4: "gemm_skinny_kernel (split-K tcgen05)",
                  5: "gemv_mma_kernel (warp-MMA GEMV, B streamed into registers)"}


def skinny_roofline(dg, ex: dict, key: str, peaks: dict) -> dict:
    """roofline-shaped entry for one decode shape, from its `extra` record."""
    name = SKINNY_ROOFLINES[key]
    rec = ex[name]
    m = int(name.split("_")[-1].split("x")[0])
    plan = dg.dg_gemm_plan(m, 12288, 4096, dg.DG_E4M3, dg.DG_BF16)
    kernel = f"{KERNEL_OF_PATH.get(plan['path'], plan['path'])}, grid {plan['grid']}"
    algo = 12288 * 4096 + m * 4096 + m * 12288 * 2
    return {"bound": "hbm", "kernel": kernel, "workload": name.replace("_", " "),
            "achieved": round(rec["GB/s"], 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(rec["GB/s"] / peaks["hbm_gbs"], 4), "us": round(rec["us"], 3),
            "us_stream": round(rec.get("us_stream", rec["us"]), 3),
            "algorithmic_bytes": algo, "traffic": recorded_traffic(name),
            "timing": "CUDA events over 250 graph-replayed back-to-back launches, weights "
                      "rotated over copies larger than 3 x L2"}


def run_kernel(args):
    """`--kernel NAME`: time one kernel workload alone (W warm-up + K timed
    launches); used for ncu captures and tile sweeps."""
    import torch

    import fp16_tensor_core_gb300 as dg
    torch.cuda.set_device(0)
    dg.dg_init()
    peaks = load_peaks()
    cases = kernel_cases(torch, dg)
    rec = measure_case(torch, dg, cases[args.kernel], torch.cuda.current_stream(), peaks,
                       args.steps, args.warmup, graph=args.graph)
    rec["kernel"] = args.kernel
    rec["force_block_n"] = os.environ.get("DG_FORCE_BLOCK_N")
    print(json.dumps(rec), flush=True)


def cpu_baseline_sample(A32, B32, sd: float, rows: int) -> dict:
    """The oracle, as it stands, on `rows` rows of A against all of B: full
    amax/scale of A and B, quantise of the sampled rows and all of B, the
    FP64 contraction and the E4M3 epilogue."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    sa = oracle.scale_from_amax(oracle.amax(A32))
    sb = oracle.scale_from_amax(oracle.amax(B32))
    qa = oracle.quantize_e4m3(A32[:rows], sa)
    qb = oracle.quantize_e4m3(B32, sb)
    R = oracle.gemm_e4m3(qa, qb, with_abs=False)
    oracle.epilogue_e4m3(R, sa, sb, np.float32(sd))
    dt = time.perf_counter() - t0
    cores = os.cpu_count() or 1
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        pass
    return {"seconds": dt, "flop": 2.0 * rows * N * K, "cores": cores}


def run_own(args):
    import numpy as np
    import torch

    import fp16_tensor_core_gb300 as dg
    import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dg.dg_init()
    peaks = load_peaks()
    sd = json.load(open(os.path.join(ROOT, "tests", "golden", "sd_8192.json")))["scale_d"]

    A32, B32 = synth.make_inputs(WORKLOAD)
    wl = Workload(torch, dg, A32, B32, sd)
    stream = torch.cuda.current_stream()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        wl.step(stream)
    torch.cuda.synchronize()
    # keep the GPU busy for ~1.5 s before the timed region so that the clock
    # sampler (100 ms period) sees the step under sustained load
    t_end = time.time() + args.settle_seconds
    while time.time() < t_end:
        wl.step(stream)
        torch.cuda.synchronize()
    st = dg.dg_sync_status()
    assert st == dg.DG_OK, dg.dg_status_string(st)

    # The GEMM's own duration comes from an event pair around it on every
    # GEMM_EVENT_EVERY-th step of the timed region: an event between two
    # kernels stops the next one from starting early (launch overlap), which
    # costs 5-10 us per step, so not every step carries the pair.
    timed = [i for i in range(args.steps) if i % GEMM_EVENT_EVERY == 0]
    evs = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for i in timed}
    barrier(world)
    torch.cuda.synchronize()
    t_s, t_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_s.record(stream)
    for i in range(args.steps):
        wl.step(stream, evs.get(i))
    t_e.record(stream)
    t_e.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_local = t_s.elapsed_time(t_e)
    gemm_ms = statistics.mean(a.elapsed_time(b) for a, b in evs.values())
    st = dg.dg_sync_status()
    assert st == dg.DG_OK, dg.dg_status_string(st)
    ms_total = reduce_max(ms_local, world, device=f"cuda:{local}")
    ms_step = ms_total / args.steps
    value = world * FLOP_PER_STEP / (ms_step * 1e-3) / 1e12

    # The same step captured once into a CUDA graph, K replays timed.
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        wl.step(torch.cuda.current_stream())
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    g_s, g_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g_s.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g_e.record(stream)
    g_e.synchronize()
    graph_ms = reduce_max(g_s.elapsed_time(g_e), world, device=f"cuda:{local}") / args.steps
    del graph
    st = dg.dg_sync_status()
    assert st == dg.DG_OK, dg.dg_status_string(st)

    # End to end: every step copies its FP32 inputs in from pinned host
    # memory and its E4M3 result back out.  Two device buffer sets let the
    # host->device copy of step i+1 and the device->host copy of step i-1
    # overlap step i's kernels (three streams, event-ordered).
    hA = torch.from_numpy(A32).pin_memory()
    hB = torch.from_numpy(B32).pin_memory()
    hD = [torch.empty((M, N), dtype=torch.uint8).pin_memory() for _ in range(2)]
    wls = [wl, Workload(torch, dg, A32, B32, sd)]
    e2e_steps = max(3, min(args.steps, 20))
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        j = i % 2
        w = wls[j]
        if i >= 2:
            s_h2d.wait_event(ev_cmp[j])      # buffer j's previous step is done
        with torch.cuda.stream(s_h2d):
            w.A.copy_(hA, non_blocking=True)
            w.B.copy_(hB, non_blocking=True)
            ev_in[j].record(s_h2d)
        stream.wait_event(ev_in[j])
        if i >= 2:
            stream.wait_event(ev_out[j])     # D of buffer j has been read out
        w.step(stream)
        ev_cmp[j].record(stream)
        s_d2h.wait_event(ev_cmp[j])
        with torch.cuda.stream(s_d2h):
            hD[j].copy_(w.D, non_blocking=True)
            ev_out[j].record(s_d2h)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_s.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    e_e.record(s_d2h)
    e_e.synchronize()
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e_s.elapsed_time(e_e), world, device=f"cuda:{local}") / e2e_steps
    st = dg.dg_sync_status()
    assert st == dg.DG_OK, dg.dg_status_string(st)

    fp8_peak = 2.0 * peaks["bf16_tflops"]
    plan = dg.dg_gemm_plan(M, N, K, dg.DG_E4M3, dg.DG_E4M3)
    achieved = FLOP_PER_STEP / (gemm_ms * 1e-3) / 1e12
    traffic = recorded_traffic("fp8_gemm_8192_e4m3out")
    line = {
        "metric": "FP8 GEMM TFLOPS (and GB/s at M=1) on 1 GB300, % of roofline",
        "value": value,
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": {
            "workload": "FP8 E4M3 GEMM 8192x8192x8192, E4M3 output, per-tensor scales",
            "M": M, "N": N, "K": K,
            "step": "amax(A), amax(B) -> scale -> quantise(A), quantise(B) -> GEMM (E4M3 out)",
            "inputs": "FP32 A, B ~ N(0,1) seed 0, resident in HBM; sD from tests/golden/sd_8192.json",
            "l2": "inputs larger than L2 (2 x 268 MB FP32 per step), no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "launch": "4 stream launches per step (graph_replay: the same step as one CUDA-graph replay)",
        },
        "roofline": {
            "bound": "tensor",
            "kernel": f"{'gemm_tc_pair_kernel' if plan['block_m'] == 256 else 'gemm_tc_kernel'} "
                      f"(tcgen05 E4M3, {plan['block_m']}x{plan['block_n']} tiles, "
                      f"{plan['stages']} stages of {plan['block_k'] // 128} K block(s), "
                      f"grid {plan['grid']})",
            "achieved": achieved,
            "peak": fp8_peak,
            "unit": "TFLOP/s",
            "frac": achieved / fp8_peak,
            "peak_source": f"{peaks['source']}: bf16 burst {peaks['bf16_tflops']} x 2 (FP8/BF16 dense ratio)",
            "frac_vs_nominal": achieved / NOMINAL_FP8_TFLOPS,
            "nominal_peak": NOMINAL_FP8_TFLOPS,
            "launch_ms": gemm_ms,
            "launch_timing": f"CUDA events around the GEMM on every {GEMM_EVENT_EVERY}th step of "
                             f"the timed region ({len(evs)} of {args.steps} steps)",
            "traffic": traffic,
        },
        "e2e": {"value": world * FLOP_PER_STEP / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "note": "pinned host FP32 inputs copied in and E4M3 D copied out every step; "
                        "copies of neighbouring steps overlap the kernels (double-buffered)",
                "h2d_bytes_per_step": A32.nbytes + B32.nbytes,
                "d2h_bytes_per_step": M * N},
        "graph_replay": {"value": world * FLOP_PER_STEP / (graph_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                         "ms_per_step": graph_ms},
        "gpu_launches": Workload.KERNELS_PER_STEP * args.steps,
        "clocks": clk,
    }
    del hA, hB, hD, wls
    skinny = {}
    if rank == 0 and not args.no_extra:
        ex = extras(torch, dg, stream, peaks)
        skinny = {k: skinny_roofline(dg, ex, k, peaks) for k in SKINNY_ROOFLINES}
        line["roofline"].update(skinny)
        line["extra"] = {k: compact(v) for k, v in ex.items()}
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline_sample(A32, B32, sd, rows=CPU_SAMPLE_ROWS)
        line["cpu_baseline"] = {
            "value": cb["flop"] / cb["seconds"] / 1e12, "unit": "TFLOPS", "cores": cb["cores"],
            "kind": "oracle", "seconds": cb["seconds"],
            "sample": f"rows 0-{CPU_SAMPLE_ROWS - 1} of A against all 8192 rows of B "
                      f"({CPU_SAMPLE_ROWS}x8192x8192): full-tensor "
                      "amax/scale of A and B, quantise of the sampled rows and all of B, FP64 "
                      "contraction, E4M3 epilogue"}
    # The decode shapes last, so that they sit in the line's tail.
    for k, v in skinny.items():
        line[f"roofline_{k}"] = v
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The oracle on the host cores, on bounded samples of the same workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np  # noqa: F401

    import synth
    sd = json.load(open(os.path.join(ROOT, "tests", "golden", "sd_8192.json")))["scale_d"]
    A32, B32 = synth.make_inputs(WORKLOAD)
    rows = 64
    for _ in range(args.warmup):
        cpu_baseline_sample(A32, B32, sd, rows)
    times, cores = [], 1
    for _ in range(args.steps):
        r = cpu_baseline_sample(A32, B32, sd, rows)
        times.append(r["seconds"])
        cores = r["cores"]
    sec = statistics.mean(times)
    value = 2.0 * rows * N * K / sec / 1e12
    sample = (f"each step: rows 0-{rows - 1} of A against all 8192 rows of B ({rows}x8192x8192): "
              "full-tensor amax/scale, quantise, FP64 contraction, E4M3 epilogue")
    line = {
        "metric": "FP8 GEMM TFLOPS (and GB/s at M=1) on 1 GB300, % of roofline",
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": "FP8 E4M3 GEMM 8192x8192x8192, E4M3 output, per-tensor scales",
                   "M": M, "N": N, "K": K, "sampled_rows": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# Kernels behind the workloads whose DRAM traffic is recorded: (name pattern
# in the ncu CSV, sources the counters depend on, algorithmic bytes per
# launch, description).
TRAFFIC_KERNELS = {
    "fp8_gemm_8192_e4m3out": ("gemm_tc_pair_kernel",
                              ["k_gemm_tc2.cu", "gemm_common.cuh", "dg_ptx.cuh"],
                              3 * 8192 * 8192, "E4M3 8192^3, E4M3 out, 256 x 256 CTA-pair tiles"),
    "qkv_gemv_1x12288x4096": ("gemv_mma_kernel", ["k_gemv_mma.cu", "dg_ptx.cuh"],
                              12288 * 4096 + 4096 + 12288 * 2,
                              "E4M3 1 x 12288 x 4096 (decode QKV), warp-MMA GEMV"),
    "qkv_m8_8x12288x4096": ("gemv_mma_kernel", ["k_gemv_mma.cu", "dg_ptx.cuh"],
                            12288 * 4096 + 8 * 4096 + 8 * 12288 * 2,
                            "E4M3 8 x 12288 x 4096, warp-MMA GEMV"),
    "qkv_m16_16x12288x4096": ("gemm_skinny_kernel",
                              ["k_gemm_skinny.cu", "gemm_common.cuh", "dg_ptx.cuh"],
                              12288 * 4096 + 16 * 4096 + 16 * 12288 * 2,
                              "E4M3 16 x 12288 x 4096, split-K tcgen05"),
}


def record_traffic(pairs):
    """`--record-traffic workload=csv ...`: records in profiles/traffic.json,
    from the CSV logs of one-pass ncu captures (dram__bytes_read.sum,
    dram__bytes_write.sum, gpu__time_duration.sum) of `--kernel workload`,
    each workload's DRAM bytes with the hash of the sources it was taken on.
    Entries of other workloads are kept."""
    import csv
    out = {"note": "one captured launch per workload after its warm-up launches; DRAM bytes "
                   "read + written per launch",
           "entries": []}
    if os.path.exists(PROFILE_TRAFFIC):
        with open(PROFILE_TRAFFIC) as f:
            out["entries"] = json.load(f).get("entries", [])
    recorded = [arg.split("=", 1)[0] for arg in pairs]
    out["entries"] = [e for e in out["entries"] if e.get("workload") not in recorded]
    for arg in pairs:
        workload, path = arg.split("=", 1)
        pattern, sources, algo, desc = TRAFFIC_KERNELS[workload]
        with open(path) as f:
            rows = list(csv.reader(line for line in f if not line.startswith("==")))
        vals = {}
        for r in rows[1:]:
            d = dict(zip(rows[0], r))
            if pattern in d.get("Kernel Name", ""):
                vals[d["Metric Name"]] = float(d["Metric Value"].replace(",", ""))
        rd, wr = int(vals["dram__bytes_read.sum"]), int(vals["dram__bytes_write.sum"])
        out["entries"].append({
            "workload": workload, "kernel": pattern, "description": desc, "sources": sources,
            "source_sha256_16": source_hash(sources), "dram_bytes_read": rd, "dram_bytes_write": wr,
            "dram_bytes_per_launch": rd + wr, "algorithmic_bytes_per_launch": algo,
            "duration_ns_under_ncu": vals.get("gpu__time_duration.sum"),
            "command": f"python bench.py --kernel {workload} --steps 2 --warmup 1 && ncu --metrics "
                       "dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
                       f"--clock-control none -k regex:{pattern} -s 1 -c 1 --csv --log-file "
                       f"traffic.csv python bench.py --kernel {workload} --steps 2 --warmup 1"})
    out["entries"].sort(key=lambda e: e["workload"])
    with open(PROFILE_TRAFFIC, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


def main(argv=None):
    args = parse_args(argv)
    if args.record_traffic:
        record_traffic(args.record_traffic)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel:
        run_kernel(args)
    else:
        run_own(args)


if __name__ == "__main__":
    main()

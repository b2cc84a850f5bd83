"""Write the stored expected values under tests/golden/ from the CPU oracle.

Calls only `oracle` (and the shared `synth` input generator).  Run from the
repository root:  python tests/golden/make_golden.py [--only sd_8192]

sd_8192.json -- the output scale of the 8192^3 E4M3-output workload:
    sD = fl32(max |Dref| / 448), Dref = sA * sB * (A_q @ B_q^T) in FP64 over
    the oracle-quantised seed-0 N(0,1) inputs (per-tensor scale = amax/448).
    [FP8-guide] ("DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南") §3.2: the output
    scale is the largest absolute output value over 448, recorded ahead of
    time; the workload supplies it precomputed.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def make_sd(name: str, out: str) -> None:
    t0 = time.time()
    A, B = synth.make_inputs(name)
    qa, sa, _ = oracle.quantize_tensor(A)
    qb, sb, _ = oracle.quantize_tensor(B)
    del A, B
    R = oracle.gemm_e4m3(qa, qb, with_abs=False)
    amax_r = float(np.max(np.abs(R)))
    dref_amax = amax_r * float(sa) * float(sb)
    sd = np.float32(dref_amax / 448.0)
    rec = {
        "workload": name,
        "shape": list(R.shape) + [int(qa.shape[1])],
        "scale_a": float(sa), "scale_b": float(sb),
        "amax_dref": dref_amax,
        "scale_d": float(sd),
        "scale_d_hex": np.float32(sd).view(np.uint32).item(),
        "cite": "[FP8-guide] §3.2: output scale = max |output| / 448, supplied precomputed",
        "seconds": round(time.time() - t0, 1),
    }
    with open(out, "w") as f:
        json.dump(rec, f, indent=1)
    print(json.dumps(rec))


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", default=None)
    args = ap.parse_args()
    if args.only in (None, "sd_8192"):
        make_sd("fp8_8192_e4m3out", os.path.join(HERE, "sd_8192.json"))


if __name__ == "__main__":
    main()

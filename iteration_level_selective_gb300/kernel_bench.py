"""Kernel-level timing through the C ABI (for roofline and ncu captures).

    python -m iteration_level_selective_gb300.kernel_bench linear --M 2048 --N 20480 --K 5120
    python -m iteration_level_selective_gb300.kernel_bench sweep

`linear` times orca_linear (the token-wise Linear of one iteration, bf16
tcgen05) with CUDA events, after warm-up, and prints achieved TFLOP/s and
algorithmic GB/s.  Inputs are random on the device.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import _orca as C
from . import build as B


def time_linear(M: int, N: int, K: int, reps: int = 20, warmup: int = 3, mode: int = C.ORCA_LINEAR_STORE):
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    A = torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16)
    W = (torch.randn((N, K), device=dev, generator=g) * 0.02).to(torch.bfloat16)
    bias = torch.zeros(N, device=dev)
    out = torch.empty((M, N), device=dev, dtype=torch.float32 if mode in (C.ORCA_LINEAR_F32OUT, C.ORCA_LINEAR_RESID)
                      else torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()

    def run():
        C.orca_linear(C.ORCA_DTYPE_BF16, mode, A.data_ptr(), W.data_ptr(), bias.data_ptr(), out.data_ptr(), M, N, K,
                      status.data_ptr(), st.cuda_stream)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        run()
    e1.record(st)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = e0.elapsed_time(e1) / reps
    flops = 2.0 * M * N * K
    byts = (M * K + N * K) * 2 + M * N * out.element_size()
    return {"M": M, "N": N, "K": K, "ms": ms, "tflops": flops / ms / 1e9, "gbs": byts / ms / 1e6}


def main():
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="cmd", required=True)
    p = sub.add_parser("linear")
    p.add_argument("--M", type=int, required=True)
    p.add_argument("--N", type=int, required=True)
    p.add_argument("--K", type=int, required=True)
    p.add_argument("--reps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    sub.add_parser("sweep")
    a = ap.parse_args()
    B.build()
    if a.cmd == "linear":
        print(json.dumps(time_linear(a.M, a.N, a.K, a.reps, a.warmup)))
    else:
        for (N, K) in ((2304, 768), (768, 768), (3072, 768), (768, 3072), (15360, 5120), (5120, 5120),
                       (20480, 5120), (5120, 20480)):
            for M in (64, 256, 2048, 8192, 25000):
                print(json.dumps(time_linear(M, N, K, reps=10)))


if __name__ == "__main__":
    main()

"""Kernel-level timing through the C ABI (for roofline and ncu captures).

    python -m iteration_level_selective_gb300.kernel_bench linear --M 2048 --N 20480 --K 5120
    python -m iteration_level_selective_gb300.kernel_bench sweep
    python -m iteration_level_selective_gb300.kernel_bench linear-graph
    python -m iteration_level_selective_gb300.kernel_bench linears-13b-mixed

`linear` times orca_linear (the token-wise Linear of one iteration, bf16
tcgen05) with CUDA events, after warm-up, and prints achieved TFLOP/s and
algorithmic GB/s.  `linear-graph` times the small-M Linears of GPT-2-small as
they run in an iteration - 20 back-to-back launches captured in a CUDA graph,
so that launch latency and programmatic dependent launch count as they do in
the engine - next to cuBLAS (torch.nn.functional.linear) captured the same
way.  `linears-13b-mixed` runs the four token-wise Linears of one layer of
the prefill-heavy 13B iteration (24,373 rows) and its LM head (256 rows),
each with the epilogue the engine uses (bf16 store, fp32 residual add, GeLU),
one warm-up and one timed launch each, for per-launch DRAM traffic captures.
Inputs are random on the device.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import _orca as C
from . import build as B


# the Linears of one layer of the prefill-heavy 13B iteration (rows of 16
# prompts U{1024..2048} + 240 decodes) and its LM head: (name, M, N, K, mode)
LINEARS_13B_MIXED = (("qkv", 24373, 15360, 5120, C.ORCA_LINEAR_STORE),
                     ("attn_out", 24373, 5120, 5120, C.ORCA_LINEAR_RESID),
                     ("fc1", 24373, 20480, 5120, C.ORCA_LINEAR_GELU),
                     ("fc2", 24373, 5120, 20480, C.ORCA_LINEAR_RESID),
                     ("lm_head", 256, 50257, 5120, C.ORCA_LINEAR_F32OUT))


def time_linear(M: int, N: int, K: int, reps: int = 20, warmup: int = 3, mode: int = C.ORCA_LINEAR_STORE,
                scratch: bool = True):
    """scratch: pass the split-K / balanced-schedule scratch the engine gives
    every Linear (64 MB); without it the kernels run data-parallel."""
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
    scr = torch.empty(64 << 20, dtype=torch.uint8, device=dev) if scratch else None

    def run():
        C.orca_linear(C.ORCA_DTYPE_BF16, mode, A.data_ptr(), W.data_ptr(), bias.data_ptr(), out.data_ptr(), M, N, K,
                      status.data_ptr(), st.cuda_stream, scratch_ptr=scr.data_ptr() if scratch else 0,
                      scratch_bytes=(64 << 20) if scratch else 0)

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


def graph_us(fn, n: int = 20, trials: int = 3) -> float:
    """Microseconds per call of fn(stream) over n calls captured in one CUDA
    graph (best of `trials` replays)."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            fn(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                fn(s)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(trials):  # replay() launches on the current stream: the events go there too
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1000.0 / n)
    return best


def time_cublas(M: int, N: int, K: int, reps: int = 20, warmup: int = 3):
    """torch.nn.functional.linear (cuBLAS, bf16 out) on the same shapes, for reference."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    A = torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16)
    W = (torch.randn((N, K), device=dev, generator=g) * 0.02).to(torch.bfloat16)
    out = torch.empty((M, N), device=dev, dtype=torch.bfloat16)
    for _ in range(warmup):
        torch.nn.functional.linear(A, W, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        torch.nn.functional.linear(A, W, out=out)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def time_linear_graph(M: int, N: int, K: int):
    """orca_linear (bf16 store epilogue with a bias) vs cuBLAS, both graph-captured."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    A = torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16)
    W = (torch.randn((N, K), device=dev, generator=g) * 0.02).to(torch.bfloat16)
    bias = torch.randn(N, device=dev, generator=g)
    out = torch.empty((M, N), device=dev, dtype=torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def ours(s):
        C.orca_linear(C.ORCA_DTYPE_BF16, C.ORCA_LINEAR_STORE, A.data_ptr(), W.data_ptr(), bias.data_ptr(),
                      out.data_ptr(), M, N, K, status.data_ptr(), s.cuda_stream)

    bias16 = bias.to(torch.bfloat16)

    def cublas(s):
        torch.nn.functional.linear(A, W, bias16, out=out)

    t_ours = graph_us(ours)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    return {"M": M, "N": N, "K": K, "ours_us": round(t_ours, 2), "cublas_us": round(graph_us(cublas), 2)}


def time_attention(batch, n_heads: int, head_dim: int, reps: int = 5, warmup: int = 2, seed: int = 0):
    """Time orca_attention on a batch [(L_i, c_i)] with random bf16 K/V slots
    laid out back to back; returns achieved algorithmic GB/s and TFLOP/s."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    row_off, slot_base, s = [0], [], 0
    for L, c in batch:
        row_off.append(row_off[-1] + L)
        slot_base.append(s)
        s += c + L
    n_slots, N, H = s, row_off[-1], n_heads * head_dim
    K = torch.randn((n_heads, n_slots, head_dim), device=dev, generator=g, dtype=torch.bfloat16)
    V = torch.randn((n_heads, n_slots, head_dim), device=dev, generator=g, dtype=torch.bfloat16)
    Q = (torch.randn((N, H), device=dev, generator=g) * 0.2).to(torch.bfloat16)
    out = torch.empty((N, H), device=dev, dtype=torch.bfloat16)
    ws_bytes = C.orca_attention_workspace_bytes(len(batch), N, n_heads, head_dim)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    ctx = [c for _, c in batch]

    def run():
        C.orca_attention(C.ORCA_DTYPE_BF16, n_heads, head_dim, n_slots, Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                         out.data_ptr(), row_off, ctx, slot_base, ws.data_ptr(), ws_bytes, status.data_ptr(),
                         st.cuda_stream)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        run()
        e1.record(st)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = sorted(times)[len(times) // 2]
    pairs = sum(L * c + L * (L + 1) // 2 for L, c in batch)
    kv_bytes = sum(c + L for L, c in batch) * 2 * H * 2
    byts = kv_bytes + 2 * N * H * 2
    flops = 4.0 * head_dim * pairs * n_heads
    return {"rows": N, "kv_gb": kv_bytes / 1e9, "ms": ms, "gbs": byts / ms / 1e6, "tflops": flops / ms / 1e9}


ATTN_CASES = {
    # 256 decoding requests, cached contexts U{1024..4096}, 13B-shaped heads (one layer)
    "c4": lambda rng: ([(1, int(c)) for c in rng.integers(1024, 4097, 256)], 40, 128),
    # a quarter of c4 (64 requests, 3.4 GB of K/V): small enough for profiler captures
    "c4_quarter": lambda rng: ([(1, int(c)) for c in rng.integers(1024, 4097, 64)], 40, 128),
    # 16 prompts U{1024..2048} + 240 decodes with contexts U{128..2048}, 13B-shaped heads
    "c5": lambda rng: ([(int(L), 0) for L in rng.integers(1024, 2049, 16)] +
                       [(1, int(c)) for c in rng.integers(128, 2049, 240)], 40, 128),
    # four prompts of 4096 tokens, 13B-shaped heads: items with 16 key tiles on average
    "long_prompts": lambda rng: ([(4096, 0)] * 4, 40, 128),
    # the 16 prompts of c5 alone (tensor-core prefill kernel only)
    "c5_prefill": lambda rng: ([(int(L), 0) for L in rng.integers(1024, 2049, 16)], 40, 128),
    # one GPT-2-small prefill of 512 tokens plus 63 decodes with contexts U{32..768}
    "gpt2_mixed": lambda rng: ([(512, 0)] + [(1, int(c)) for c in rng.integers(32, 769, 63)], 12, 64),
    # a decode-only GPT-2-small iteration: 30 decodes with contexts U{32..768}
    "gpt2_decode": lambda rng: ([(1, int(c)) for c in rng.integers(32, 769, 30)], 12, 64),
}


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
    sub.add_parser("linear-graph")
    sub.add_parser("linears-13b-mixed")
    sub.add_parser("linear-13b")
    pa = sub.add_parser("attention")
    pa.add_argument("--case", choices=sorted(ATTN_CASES), required=True)
    pa.add_argument("--reps", type=int, default=5)
    a = ap.parse_args()
    B.build()
    if a.cmd == "attention":
        import numpy as np
        batch, nh, d = ATTN_CASES[a.case](np.random.default_rng(0))
        r = time_attention(batch, nh, d, reps=a.reps)
        r["case"] = a.case
        print(json.dumps(r))
    elif a.cmd == "linear":
        print(json.dumps(time_linear(a.M, a.N, a.K, a.reps, a.warmup)))
    elif a.cmd == "linear-13b":
        # the 13B Linears (QKV, Attn-Out, FC1, FC2) at the row counts of decode-heavy iterations
        for M in (1, 64, 128, 200, 256, 300, 384, 512, 700, 1024, 2048, 24373):
            for (N, K) in ((15360, 5120), (5120, 5120), (20480, 5120), (5120, 20480), (50257, 5120)):
                if M == 24373 and N == 50257:
                    continue
                r = time_linear(M, N, K, reps=20)
                r["no_scratch_ms"] = time_linear(M, N, K, reps=20, scratch=False)["ms"]
                r["cublas_ms"] = time_cublas(M, N, K)
                r["weight_gbs"] = N * K * 2 / r["ms"] / 1e6
                r["cublas_weight_gbs"] = N * K * 2 / r["cublas_ms"] / 1e6
                print(json.dumps(r), flush=True)
    elif a.cmd == "linears-13b-mixed":
        for name, M, N, K, mode in LINEARS_13B_MIXED:
            r = time_linear(M, N, K, reps=1, warmup=1, mode=mode)
            r["name"] = name
            print(json.dumps(r), flush=True)
            torch.cuda.empty_cache()
    elif a.cmd == "linear-graph":
        # GPT-2-small's Linears (QKV, Attn-Out, FC1, FC2, LM head) at decode and prefill row counts
        for M in (8, 64, 128, 256):
            for (N, K) in ((2304, 768), (768, 768), (3072, 768), (768, 3072), (50304, 768)):
                print(json.dumps(time_linear_graph(M, N, K)))
    else:
        for (N, K) in ((2304, 768), (768, 768), (3072, 768), (768, 3072), (15360, 5120), (5120, 5120),
                       (20480, 5120), (5120, 20480)):
            for M in (64, 256, 2048, 8192, 25000):
                print(json.dumps(time_linear(M, N, K, reps=10)))


if __name__ == "__main__":
    main()

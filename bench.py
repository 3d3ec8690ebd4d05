#!/usr/bin/env python3
"""Throughput of selectively batched iterations on one GB300 (or N replicas).

Workload (default): a GPT-2-small-shaped bf16 decoder (12 layers, H=768,
12 heads, vocab 50257, random-init N(0, 0.02) weights) serving a synthetic
trace of 64 requests - prompts U{32..512}, outputs U{1..256}, max_tokens =
prompt + 256, Poisson arrivals (0.5 per iteration), no EOS - with
iteration-level scheduling (max_bs 64, K/V slots sized to 40 GB).  One step
is one selectively batched iteration: Select, the ragged descriptor, the
whole forward over the [sum L_i, H] rows, the LM head on each request's last
row, greedy argmax and the post-iteration update.  When the trace completes
it restarts (every request fresh, all slots released).

value  = processed tokens (sum L_i) per second over the K timed iterations,
         CUDA events on the iteration stream around the timed region;
e2e    = the same through the C ABI with host request buffers, wall clock
         (host scheduling, descriptor H2D and token D2H included).
The roofline object describes the dominant kernel, timed per launch with CUDA
events in a second, profiled pass over the same iterations.

--impl reference times the CPU oracle (per-request, token-at-a-time
generation in float64) on the same trace and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "tokens/s per selective-batched iteration at 1 GB300; % of HBM/tensor roofline"
UNIT = "tokens/s"
WORKLOAD = "gpt2-small bf16, 64-request Poisson trace (prompt U32-512, out U1-256, max_tokens=prompt+256), max_bs 64"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def trace_for(rank: int, gen: int = 0):
    """The rank's request stream (replicas serve distinct streams)."""
    shape = synth.GPT2_SMALL
    return synth.make_trace(64, (32, 512), (1, 256), vocab=shape.vocab, seed=1000 * rank + gen,
                            rate_per_iter=0.5, max_extra=256)


def n_slots_for(shape) -> int:
    return int(40e9 // (shape.n_layers * 2 * shape.hidden * 2))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def kernel_source_hash() -> str:
    from iteration_level_selective_gb300.ncu_summary import source_hash
    return source_hash(os.path.join(ROOT, "iteration_level_selective_gb300", "csrc"))


def measured_traffic(kernel: str, config: str = "gpt2-trace"):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel sources and this workload (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(config, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("bytes_per_launch")


def cpu_oracle_sample(budget_s: float, rank: int = 0):
    """The oracle as it stands, on the benchmark trace: requests in arrival
    order, each generated alone token by token, until the time budget is
    spent.  Returns (tokens processed, seconds, description)."""
    from oracle import model as omodel
    shape = synth.GPT2_SMALL
    w = synth.make_weights(shape, seed=0)
    orc = omodel.GPTOracle(shape, w)
    trace = sorted(trace_for(rank), key=lambda r: (r.arrival, r.req_id))
    n_tok, n_req = 0, 0
    t0 = time.perf_counter()
    for req in trace:
        cache = orc.new_cache(req.n_prompt + req.out_len)
        last = None
        for t, tok in enumerate(req.prompt):
            last = orc.step(cache, int(tok), t, want_logits=(t == req.n_prompt - 1))
            n_tok += 1
            if time.perf_counter() - t0 > budget_s:
                break
        else:
            for k in range(1, req.out_len):
                tok = int(np.argmax(last))
                last = orc.step(cache, tok, req.n_prompt + k - 1)
                n_tok += 1
                if time.perf_counter() - t0 > budget_s:
                    break
        n_req += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return n_tok, dt, (f"oracle (float64 numpy, token-at-a-time) on the first {n_req} request(s) of the trace: "
                       f"{n_tok} tokens in {dt:.1f} s")


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return 0
    steps = args.steps if args.steps is not None else DEFAULT_STEPS["gpt2-trace"]
    # each step: the oracle processes a bounded sample of 4 token rows of the trace
    from oracle import model as omodel
    shape = synth.GPT2_SMALL
    w = synth.make_weights(shape, seed=0)
    orc = omodel.GPTOracle(shape, w)
    trace = sorted(trace_for(0), key=lambda r: (r.arrival, r.req_id))
    state = {"req": 0, "t": 0, "cache": None, "last": None}

    def one_row():
        req = trace[state["req"] % len(trace)]
        if state["cache"] is None:
            state["cache"] = orc.new_cache(req.n_prompt + req.out_len)
            state["t"] = 0
        t = state["t"]
        tok = int(req.prompt[t]) if t < req.n_prompt else int(np.argmax(state["last"]))
        state["last"] = orc.step(state["cache"], tok, t, want_logits=(t >= req.n_prompt - 1))
        state["t"] += 1
        if state["t"] >= req.n_prompt + req.out_len - 1:
            state["req"] += 1
            state["cache"] = None

    rows_per_step = 4
    for _ in range(args.warmup):
        for _ in range(rows_per_step):
            one_row()
    t0 = time.perf_counter()
    for _ in range(steps):
        for _ in range(rows_per_step):
            one_row()
    dt = time.perf_counter() - t0
    value = rows_per_step * steps / dt
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "step": f"{rows_per_step} token rows"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{rows_per_step * steps} token rows of the trace, token-at-a-time"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


CONFIGS = ("gpt2-trace", "13b-mixed", "13b-decode")
DEFAULT_STEPS = {"gpt2-trace": 200, "13b-mixed": 10, "13b-decode": 50}


def fixed_batch_spec(name: str):
    """The two fixed 13B-shaped iterations: (shape, prompt lengths, decode
    contexts, workload description)."""
    if name == "13b-mixed":
        prompts, ctx = synth.mixed_batch_lengths(16, (1024, 2048), 240, (128, 2048), seed=0)
        return (synth.GPT_13B, prompts, ctx,
                "13B-shaped bf16 (40L, H5120, 40 heads, FFN 4H, V50257), one prefill-heavy mixed iteration repeated: "
                "16 prompts U1024-2048 + 240 decodes with contexts U128-2048, max_bs 256")
    if name == "13b-decode":
        _, ctx = synth.mixed_batch_lengths(0, (1, 1), 256, (1024, 4096), seed=0)
        shape = synth.with_layers(synth.GPT_13B, 16)
        return (shape, np.zeros(0, np.int64), ctx,
                "13B-shaped bf16 with 16 of its 40 layers (the K/V of 40 layers does not fit in HBM), one "
                "decode-only iteration repeated: 256 decodes with contexts U1024-4096, max_bs 256")
    raise ValueError(name)


class TraceWorkload:
    """The GPT-2-small serving trace, restarted whenever it completes
    (optionally with chunked prefill under a per-iteration token budget)."""

    def __init__(self, eng, rank, stream, token_budget=None, chunk=None, n_workers=1):
        from iteration_level_selective_gb300 import runtime as rt
        self.rt, self.eng, self.rank, self.stream, self.gen = rt, eng, rank, stream, 0
        self.budget = (token_budget, chunk)
        self.n_workers = n_workers
        self.loop = self._new()

    def _new(self):
        self.gen += 1
        return self.rt.ServingLoop(self.eng, self.rt.RequestPool(trace_for(self.rank, self.gen)), stream=self.stream,
                                   token_budget=self.budget[0], chunk=self.budget[1], n_workers=self.n_workers)

    def step(self):
        if self.loop.done():
            self.loop = self._new()
        return self.loop.step()


class FixedBatchWorkload:
    """One selectively batched iteration, repeated.  Every request holds its
    max_tokens reservation from the start and is in the increment state:
    prompts have nothing cached (L_i = prompt length), decodes have c_i cached
    tokens (L_i = 1).  After each iteration the request counters are put
    back, so every step runs the same batch and rewrites the same K/V slots."""

    def __init__(self, eng, prompts, ctx, vocab, stream):
        from iteration_level_selective_gb300 import _orca as C
        from iteration_level_selective_gb300 import runtime as rt
        reqs = []
        for i, L in enumerate(prompts):
            reqs.append(synth.Request(req_id=i, arrival=0, prompt=synth.token_ids(int(L), vocab, stream=i),
                                      out_len=4, max_tokens=int(L) + 3))
        for j, c in enumerate(ctx):
            k = len(prompts) + j
            reqs.append(synth.Request(req_id=k, arrival=0, prompt=synth.token_ids(int(c), vocab, stream=k),
                                      out_len=4, max_tokens=int(c) + 3))
        self.pool = rt.RequestPool(reqs)
        v = self.pool.view
        for k in range(self.pool.n):
            v["slot_base"][k] = C.orca_kv_reserve(eng.handle, int(v["req_id"][k]), int(v["max_tokens"][k]))
        v["state"] = C.ORCA_INCREMENT
        v["n_cached"][len(prompts):] = ctx
        v["n_generated"][len(prompts):] = 1
        self.saved = {f: v[f].copy() for f in ("state", "n_cached", "n_generated")}
        self.loop = rt.ServingLoop(eng, self.pool, stream=stream)

    @staticmethod
    def slots_needed(prompts, ctx) -> int:
        return int(np.sum(prompts + 3) + np.sum(ctx + 3))

    def step(self):
        rec = self.loop.step()
        v = self.pool.view
        for f, a in self.saved.items():
            v[f] = a
        return rec


def run_ours(args, rank: int, world: int):
    import torch
    import torch.distributed as dist
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import build as B
    from iteration_level_selective_gb300 import replicas
    from iteration_level_selective_gb300 import runtime as rt

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    stream = torch.cuda.Stream(dev)
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[args.config]
    if args.config == "gpt2-trace":
        shape = synth.GPT2_SMALL
        host_w = synth.make_weights(shape, seed=0)
        weights = rt.DeviceWeights(shape, dev, host=host_w)
        del host_w
        n_slots = args.kv_slots if args.kv_slots else n_slots_for(shape)
        if args.reserve == "paged":
            n_slots -= n_slots % 32   # whole K/V blocks
        eng = rt.Engine(shape, weights, max_bs=64, n_slots=n_slots, max_rows=64 * 512, device=dev,
                        reserve_policy=rt.RESERVE_POLICIES[args.reserve])
        work = TraceWorkload(eng, rank, stream, args.token_budget, args.chunk, args.workers)
        workload = WORKLOAD
        if args.token_budget or args.chunk:
            workload += f", chunked prefill (token budget {args.token_budget or 'none'}, chunk {args.chunk or 'none'})"
        cfg_extra = {"model": "gpt2-small-shaped (12L, H768, 12 heads, V50257), random init", "max_bs": 64,
                     "n_slots": n_slots, "arrivals": "Poisson 0.5 per iteration",
                     "l2": "inputs larger than L2 (0.25 GB weights + K/V pool), no flush"}
        if args.token_budget or args.chunk:
            cfg_extra["token_budget"] = args.token_budget or None
            cfg_extra["chunk"] = args.chunk or None
        if args.workers != 1:
            cfg_extra["n_workers"] = args.workers
            workload += f", {args.workers} batches in flight"
        if args.reserve != "max":
            cfg_extra["reserve_policy"] = args.reserve
            workload += f", {args.reserve} K/V reservation"
    else:
        shape, prompts, ctx, workload = fixed_batch_spec(args.config)
        n_slots = FixedBatchWorkload.slots_needed(prompts, ctx)
        n_rows = int(np.sum(prompts) + len(ctx))
        weights = rt.DeviceWeights(shape, dev, host=None, seed=0)
        free, _ = torch.cuda.mem_get_info(dev)
        cfg = rt.make_config(shape, 256, n_slots, n_rows)
        need = C.orca_kv_pool_bytes(cfg) + C.orca_workspace_bytes(cfg)
        if need > free:
            raise SystemExit(f"{args.config}: K/V pool + workspace need {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free")
        eng = rt.Engine(shape, weights, max_bs=256, n_slots=n_slots, max_rows=n_rows, device=dev)
        eng.kv.zero_()   # no stale bits in the cached contexts
        work = FixedBatchWorkload(eng, prompts, ctx, shape.vocab, stream)
        cfg_extra = {"model": f"13B-shaped, {shape.n_layers} layers, random init N(0, 0.02)", "max_bs": 256,
                     "n_rows": n_rows, "n_slots": n_slots, "kv_pool_gb": round(eng.kv_bytes / 1e9, 1),
                     "weights_gb": round(weights.nbytes / 1e9, 1),
                     "l2": "inputs larger than L2 (weights and K/V many times L2), no flush"}

    def step():
        rec = work.step()
        h2d, d2h, _ = C.orca_last_transfer(eng.handle)
        return rec, h2d, d2h

    def kv_usage():
        pool = work.loop.pool if hasattr(work, "loop") else work.pool
        return C.orca_kv_usage(eng.handle, pool.arr, pool.n)

    warmup = max(3, args.warmup)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rows = gen_tok = done = h2d = d2h = launches = 0
    step_ms, usage = [], []
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    ev0.record(stream)
    for _ in range(steps):
        t0 = time.perf_counter()
        rec, hb, db = step()
        step_ms.append(1000.0 * (time.perf_counter() - t0))
        usage.append(kv_usage())
        rows += sum(rec.n_new)
        gen_tok += sum(1 for t in rec.next_tokens if t >= 0)
        done += len(rec.released)
        h2d += hb
        d2h += db
        launches += rec.launches
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - w0
    clocks = sampler.stop()
    dev_s = ev0.elapsed_time(ev1) / 1000.0
    (dev_s, wall), (rows, gen_tok, done, h2d, d2h, launches) = replicas.reduce_timing(
        [dev_s, wall], [rows, gen_tok, done, h2d, d2h, launches], device=dev)

    # profiled pass: per-launch CUDA events around every kernel, same workload
    C.orca_profile_enable(eng.handle, True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    stats = {C.KERNEL_NAMES[k]: C.orca_profile_read(eng.handle, k) for k in range(C.ORCA_K_COUNT)}
    C.orca_profile_enable(eng.handle, False)
    kernels = {
        "gemm_tc_bf16": [stats[n] for n in ("gemm_qkv", "gemm_o", "gemm_fc1", "gemm_fc2", "lm_head")],
        "attention": [stats["attention"]],
        "layernorm": [stats["layernorm"]],
        "embed": [stats["embed"]],
        "argmax": [stats["argmax"]],
    }
    agg = {}
    for k, lst in kernels.items():
        agg[k] = {"launches": sum(s["launches"] for s in lst), "ms": sum(s["total_ms"] for s in lst),
                  "flops": sum(s["flops"] for s in lst), "bytes": sum(s["bytes"] for s in lst)}
    total_ms = sum(a["ms"] for a in agg.values()) or 1.0
    dom = max(agg, key=lambda k: agg[k]["ms"])
    a = agg[dom]
    peaks, peak_src = load_peaks()
    balance = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if a["bytes"] > 0 and a["flops"] / a["bytes"] > balance:
        achieved = a["flops"] / (a["ms"] / 1000.0) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s"}
    else:
        achieved = a["bytes"] / (a["ms"] / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(dom, args.config)
    roof["kernel"] = dom
    roof["peak_source"] = peak_src + (" sustained bf16" if roof["bound"] == "tensor" else " copy bandwidth")
    roof["launches"] = a["launches"]
    roof["algorithmic_per_launch"] = (a["flops"] if roof["bound"] == "tensor" else a["bytes"]) / max(1, a["launches"])
    # the other kernel classes against their own bound
    per_kernel = {}
    for k, v in agg.items():
        if v["ms"] <= 0:
            continue
        if v["bytes"] > 0 and v["flops"] / v["bytes"] > balance:
            per_kernel[k] = {"TFLOP/s": round(v["flops"] / v["ms"] / 1e9, 1),
                             "frac_tensor": round(v["flops"] / v["ms"] / 1e9 / peaks["bf16_tflops_sustained"], 3)}
        else:
            per_kernel[k] = {"GB/s": round(v["bytes"] / v["ms"] / 1e6, 1),
                             "frac_hbm": round(v["bytes"] / v["ms"] / 1e6 / peaks["hbm_gbs"], 3)}
    value = rows / dev_s
    config = {"workload": workload}
    config.update(cfg_extra)
    config["parallelism"] = f"replicas x{world}"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": 1000.0 * dev_s / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "generated_tokens_per_s": gen_tok / dev_s,
        "completed_requests_per_s": done / dev_s,
        "e2e": {"value": rows / wall, "unit": UNIT, "h2d_bytes_per_step": h2d / steps / max(1, world),
                "d2h_bytes_per_step": d2h / steps / max(1, world)},
        "gpu_launches": launches,
        "kv_usage": {"reserved_frac": round(float(np.mean([u[0] for u in usage])) / n_slots, 5),
                     "stored_frac": round(float(np.mean([u[1] for u in usage])) / n_slots, 5),
                     "stored_over_reserved": round(float(np.sum([u[1] for u in usage]) /
                                                         max(1, np.sum([u[0] for u in usage]))), 4),
                     "weighting": "per iteration, after each timed iteration"},
        "generated_per_iteration": round(gen_tok / steps / max(1, world), 2),
        "iteration_ms": {"p50": round(float(np.percentile(step_ms, 50)), 4),
                         "p99": round(float(np.percentile(step_ms, 99)), 4), "max": round(max(step_ms), 4),
                         "clock": "host wall clock per iteration (the call waits for the tokens)"},
        "roofline": roof,
        "kernel_roofline": per_kernel,
        "kernel_time_share": {k: round(v["ms"] / total_ms, 4) for k, v in agg.items()},
        "kernel_ms_per_step": {k: round(v["ms"] / steps, 4) for k, v in agg.items()},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if args.config == "gpt2-trace":
            n_tok, dt, desc = cpu_oracle_sample(args.cpu_seconds)
            line["cpu_baseline"] = {"value": n_tok / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": desc}
        else:
            line["cpu_baseline"] = None
            line["cpu_baseline_note"] = ("the float64 oracle needs the 13B weights on the host (50 GB in float64 "
                                         "per 40 layers); it is timed on the GPT-2-small trace only")
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed iterations (default: 200 for gpt2-trace, 10 for 13b-mixed, 50 for 13b-decode)")
    ap.add_argument("--config", choices=CONFIGS, default="gpt2-trace",
                    help="gpt2-trace (the serving trace, default), 13b-mixed (one prefill-heavy 13B iteration), "
                         "13b-decode (one decode-only 13B iteration)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--token-budget", type=int, default=0,
                    help="gpt2-trace only: chunked prefill with this many rows per iteration at most")
    ap.add_argument("--chunk", type=int, default=0,
                    help="gpt2-trace only: prompt chunk size for chunked prefill")
    ap.add_argument("--workers", type=int, choices=[1, 2], default=1,
                    help="gpt2-trace only: batches in flight at once (Algorithm 1's n_workers)")
    ap.add_argument("--reserve", choices=["max", "pow2", "oracle", "paged"], default="max",
                    help="gpt2-trace only: K/V reservation policy (max_tokens, power of two, true length) or "
                         "paged K/V (32-slot blocks on demand, preemption of the latest arrival)")
    ap.add_argument("--kv-slots", type=int, default=0,
                    help="gpt2-trace only: K/V pool slots (default: 40 GB worth); the trace needs at most "
                         "64 x 768, so profiler captures use a small pool")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
    else:
        rc = run_ours(args, rank, world)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())

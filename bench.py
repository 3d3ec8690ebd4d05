#!/usr/bin/env python3
"""Throughput of selectively batched iterations on one GB300 (or N replicas).

Default workload (--config 13b-mixed): a 13B-shaped bf16 decoder (40 layers,
H=5120, 40 heads of 128, FFN 4H, vocab 50257, random-init N(0, 0.02)
weights) running one prefill-heavy mixed iteration - 16 prompts of
U{1024..2048} tokens next to 240 decoding requests with U{128..2048} cached
tokens, about 24k rows, max_bs 256 - repeated.  One step is one selectively
batched iteration: Select, the ragged descriptor, the whole forward over the
[sum L_i, H] rows, the LM head on each request's last row, greedy argmax and
the post-iteration update.  The same line carries the decode-dominated
iteration (256 decodes with U{1024..4096} cached tokens, 16 of the 40 layers
because 40 layers of that K/V exceed HBM) as `decode_stress`.

Other workloads: --config 13b-decode (that decode iteration alone),
--config 13b-trace (the 13B serving trace: 1024 requests, input and output
U{32..512}, Poisson arrivals, max_bs 256, 120 GB of K/V reservations) and
--config gpt2-trace (a GPT-2-small-shaped model serving 64 requests).  A
trace run times whole traces and reports overall and steady-state figures.

value  = processed tokens (sum L_i) per second over the timed iterations,
         CUDA events on the iteration stream around the timed region;
e2e    = the same through the C ABI with host request buffers, wall clock
         (host scheduling, descriptor H2D and token D2H included);
roofline = the dominant kernel class, timed per launch on the same path: the
         timed iterations replayed again with launch stamps (every kernel
         raises a %globaltimer end stamp; a launch's share is its end minus
         the previous launch's end), with a CUDA-event pass as a cross-check;
iteration_roofline = max(weight + K/V bytes at the HBM peak, FLOPs at the
         tensor peak) over the measured iteration time.

--impl reference times the CPU oracle (per-request, token-at-a-time
generation in float64) on the same workload and metric.
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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

CONFIGS = ("13b-mixed", "13b-decode", "13b-trace", "gpt2-trace")
DEFAULT_CONFIG = "13b-mixed"
# timed iterations of the fixed-batch workloads; trace workloads time whole traces
DEFAULT_STEPS = {"13b-mixed": 10, "13b-decode": 50, "13b-trace": 1, "gpt2-trace": 1}
TRACES = ("13b-trace", "gpt2-trace")

GPT2_WORKLOAD = ("gpt2-small-shaped bf16 (12L, H768, 12 heads, V50257), 64-request Poisson trace (prompt U32-512, "
                 "out U1-256, max_tokens=prompt+256, 0.5 arrivals per iteration), max_bs 64")
T13B_WORKLOAD = ("13B-shaped bf16 (40L, H5120, 40 heads, FFN 4H, V50257), 1024-request Poisson trace (input U32-512, "
                 "output U32-512, max_tokens=input+output, 1 arrival per iteration), max_bs 256, K/V slots for 120 GB")


# ------------------------------------------------------------------ workloads

def gpt2_trace(rank: int, gen: int = 0):
    """The rank's GPT-2-small request stream (replicas serve distinct streams)."""
    return synth.make_trace(64, (32, 512), (1, 256), vocab=synth.GPT2_SMALL.vocab, seed=1000 * rank + gen,
                            rate_per_iter=0.5, max_extra=256)


def trace_13b(rank: int, gen: int = 0):
    """The 13B serving trace: max_tokens = input + output (no EOS, so the
    output length is the most a request generates)."""
    return synth.make_trace(1024, (32, 512), (32, 512), vocab=synth.GPT_13B.vocab, seed=7000 + 1000 * rank + gen,
                            rate_per_iter=1.0)


def trace_spec(name: str):
    """(shape, trace factory, max_bs, n_slots, max_rows, description)."""
    if name == "gpt2-trace":
        s = synth.GPT2_SMALL
        return s, gpt2_trace, 64, int(40e9 // (s.n_layers * 2 * s.hidden * 2)), 64 * 512, GPT2_WORKLOAD
    if name == "13b-trace":
        s = synth.GPT_13B
        return s, trace_13b, 256, int(120e9 // (s.n_layers * 2 * s.hidden * 2)), 256 * 512, T13B_WORKLOAD
    raise ValueError(name)


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
    """A serving trace under iteration-level scheduling, run to completion
    (optionally with chunked prefill under a per-iteration token budget)."""

    def __init__(self, eng, trace, stream, token_budget=None, chunk=None, n_workers=1):
        from iteration_level_selective_gb300 import runtime as rt
        self.pool = rt.RequestPool(trace)
        self.loop = rt.ServingLoop(eng, self.pool, stream=stream, token_budget=token_budget, chunk=chunk,
                                   n_workers=n_workers)

    def done(self):
        return self.loop.done()

    def step(self):
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

    def done(self):
        return False

    def step(self):
        rec = self.loop.step()
        v = self.pool.view
        for f, a in self.saved.items():
            v[f] = a
        return rec


# ------------------------------------------------------------------ measurement helpers

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


def measured_traffic(kernel: str, config: str):
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


def iteration_work(shape, batch, elem_bytes: int = 2):
    """Algorithmic work of one iteration over batch = [(L_i, c_i)]: Linear,
    LM head and attention FLOPs, and the K/V bytes read (cached tokens) and
    written (new rows), all layers."""
    H, nL, V = shape.hidden, shape.n_layers, shape.vocab
    N = sum(L for L, _ in batch)
    B = len(batch)
    pairs = sum(L * c + L * (L + 1) // 2 for L, c in batch)   # keys each new row attends over
    cached = sum(c for _, c in batch)
    flops = 2.0 * N * 12 * H * H * nL + 2.0 * B * H * V + 4.0 * H * pairs * nL
    kv_bytes = (cached + N) * 2.0 * H * elem_bytes * nL
    return flops, kv_bytes


def iteration_roofline(shape, weight_bytes: float, batches, measured_s: float, peaks):
    """Sum over iterations of max((weights + K/V bytes) / HBM peak, FLOPs /
    sustained bf16 peak), against the measured time of those iterations."""
    bw = peaks["hbm_gbs"] * 1e9
    tp = peaks["bf16_tflops_sustained"] * 1e12
    t_roof = t_mem = t_flop = flops = kvb = 0.0
    for batch in batches:
        f, kv = iteration_work(shape, batch)
        tm, tf = (weight_bytes + kv) / bw, f / tp
        t_roof += max(tm, tf)
        t_mem += tm
        t_flop += tf
        flops += f
        kvb += kv
    n = max(1, len(batches))
    return {"frac": t_roof / measured_s if measured_s > 0 else None,
            "t_roof_ms_per_step": 1000 * t_roof / n, "t_measured_ms_per_step": 1000 * measured_s / n,
            "bound": "tensor" if t_flop >= t_mem else "hbm",
            "flops_per_step": flops / n, "weight_bytes": weight_bytes, "kv_bytes_per_step": kvb / n,
            "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops_sustained": peaks["bf16_tflops_sustained"]}}


def kernel_classes(C, eng):
    stats = {C.KERNEL_NAMES[k]: C.orca_profile_read(eng.handle, k) for k in range(C.ORCA_K_COUNT)}
    groups = {
        "gemm_tc_bf16": ("gemm_qkv", "gemm_o", "gemm_fc1", "gemm_fc2", "lm_head"),
        "attention": ("attention",), "layernorm": ("layernorm",), "embed": ("embed",), "argmax": ("argmax",),
    }
    agg = {}
    for k, names in groups.items():
        lst = [stats[n] for n in names]
        agg[k] = {"launches": sum(s["launches"] for s in lst), "ms": sum(s["total_ms"] for s in lst),
                  "flops": sum(s["flops"] for s in lst), "bytes": sum(s["bytes"] for s in lst)}
    return agg


def roofline_of(agg, kernel, peaks, peak_src, config):
    """Roofline object of one kernel class: tensor-bound when its algorithmic
    intensity is above the ridge of the measured peaks, else HBM-bound."""
    a = agg[kernel]
    balance = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if a["bytes"] > 0 and a["flops"] / a["bytes"] > balance:
        roof = {"bound": "tensor", "achieved": a["flops"] / (a["ms"] / 1000.0) / 1e12,
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": a["bytes"] / (a["ms"] / 1000.0) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(kernel, config)
    roof["kernel"] = kernel
    roof["peak_source"] = peak_src + (" sustained bf16" if roof["bound"] == "tensor" else " copy bandwidth")
    roof["launches"] = a["launches"]
    roof["algorithmic_per_launch"] = (a["flops"] if roof["bound"] == "tensor" else a["bytes"]) / max(1, a["launches"])
    roof["ms_per_launch"] = a["ms"] / max(1, a["launches"])
    return roof


def per_kernel_roofline(agg, peaks):
    balance = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    out = {}
    for k, v in agg.items():
        if v["ms"] <= 0:
            continue
        if v["bytes"] > 0 and v["flops"] / v["bytes"] > balance:
            out[k] = {"TFLOP/s": round(v["flops"] / v["ms"] / 1e9, 1),
                      "frac_tensor": round(v["flops"] / v["ms"] / 1e9 / peaks["bf16_tflops_sustained"], 3)}
        else:
            out[k] = {"GB/s": round(v["bytes"] / v["ms"] / 1e6, 1),
                      "frac_hbm": round(v["bytes"] / v["ms"] / 1e6 / peaks["hbm_gbs"], 3)}
    return out


# ------------------------------------------------------------------ CPU oracle samples

def oracle_13b_slice(n_layers: int = 2):
    """The oracle on the first layers of the 13B shape (the float64 weights of
    all 40 layers, 100 GB, do not fit a host budget)."""
    from oracle import model as omodel
    shape = synth.with_layers(synth.GPT_13B, n_layers)
    return omodel.GPTOracle(shape, synth.make_weights(shape, seed=0)), shape


def cpu_oracle_sample(config: str, budget_s: float):
    """The oracle as it stands on the workload's requests, each generated
    alone token by token, until the time budget is spent.  Returns (tokens/s
    for the workload's model, description)."""
    if config.startswith("13b"):
        orc, shape = oracle_13b_slice()
        scale = shape.n_layers / synth.GPT_13B.n_layers if config != "13b-decode" else shape.n_layers / 16
        prompts, ctx = fixed_batch_spec(config)[1:3] if config != "13b-trace" else (np.array([512]), [])
        lengths = [int(L) for L in prompts] + [int(c) for c in ctx]
        model = "2-layer slice of the 13B shape"
    else:
        from oracle import model as omodel
        shape = synth.GPT2_SMALL
        orc = omodel.GPTOracle(shape, synth.make_weights(shape, seed=0))
        scale = 1.0
        lengths = [r.n_prompt for r in sorted(gpt2_trace(0), key=lambda r: (r.arrival, r.req_id))]
        model = "GPT-2-small shape, all 12 layers"
    n_tok, n_req = 0, 0
    t0 = time.perf_counter()
    for i, L in enumerate(lengths):
        toks = synth.token_ids(L, shape.vocab, stream=i)
        cache = orc.new_cache(L + 1)
        for t, tok in enumerate(toks):
            orc.step(cache, int(tok), t, want_logits=(t == L - 1))
            n_tok += 1
            if time.perf_counter() - t0 > budget_s:
                break
        n_req += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    value = n_tok / dt * scale
    desc = (f"oracle (float64 numpy, token-at-a-time) on the {model}: {n_tok} tokens of {n_req} request(s) of the "
            f"workload in {dt:.1f} s")
    if scale != 1.0:
        desc += f"; tokens/s scaled by {scale:.3f} (layers of the slice / layers of the timed model)"
    return value, desc


def run_reference(args, rank: int, world: int):
    """The oracle as the reference arm: each step feeds a bounded sample of
    the workload's token rows to the oracle, one token at a time."""
    if rank != 0:
        return 0
    config = args.config
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[config]
    if config.startswith("13b"):
        orc, shape = oracle_13b_slice()
        scale = shape.n_layers / (16 if config == "13b-decode" else synth.GPT_13B.n_layers)
        rows_per_step = 2
        model = "2-layer slice of the 13B shape, scaled to the timed layer count"
    else:
        from oracle import model as omodel
        shape = synth.GPT2_SMALL
        orc = omodel.GPTOracle(shape, synth.make_weights(shape, seed=0))
        scale = 1.0
        rows_per_step = 4
        model = "GPT-2-small shape"
    toks = synth.token_ids(4096, shape.vocab, stream=0)
    state = {"t": 0, "cache": orc.new_cache(4096)}

    def one_row():
        t = state["t"]
        if t == 4096:
            state["t"], state["cache"] = 0, orc.new_cache(4096)
            t = 0
        orc.step(state["cache"], int(toks[t]), t, want_logits=False)
        state["t"] += 1

    for _ in range(args.warmup):
        for _ in range(rows_per_step):
            one_row()
    t0 = time.perf_counter()
    for _ in range(steps):
        for _ in range(rows_per_step):
            one_row()
    dt = time.perf_counter() - t0
    value = rows_per_step * steps / dt * scale
    cores = os.cpu_count()
    workload = (fixed_batch_spec(config)[3] if config in ("13b-mixed", "13b-decode") else trace_spec(config)[5])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload, "step": f"{rows_per_step} token rows"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{rows_per_step * steps} token rows fed one at a time, {model}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def _free_engine(eng, weights):
    import torch
    eng.close()
    del eng.kv, eng.ws
    weights.tensors.clear()
    torch.cuda.empty_cache()


def build_fixed(config, dev, stream):
    import torch
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import runtime as rt
    shape, prompts, ctx, workload = fixed_batch_spec(config)
    n_slots = FixedBatchWorkload.slots_needed(prompts, ctx)
    n_rows = int(np.sum(prompts) + len(ctx))
    weights = rt.DeviceWeights(shape, dev, host=None, seed=0)
    free, _ = torch.cuda.mem_get_info(dev)
    cfg = rt.make_config(shape, 256, n_slots, n_rows)
    need = C.orca_kv_pool_bytes(cfg) + C.orca_workspace_bytes(cfg)
    if need > free:
        raise SystemExit(f"{config}: K/V pool + workspace need {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free")
    eng = rt.Engine(shape, weights, max_bs=256, n_slots=n_slots, max_rows=n_rows, device=dev)
    eng.kv.zero_()   # no stale bits in the cached contexts
    work = FixedBatchWorkload(eng, prompts, ctx, shape.vocab, stream)
    extra = {"model": f"13B-shaped, {shape.n_layers} layers, random init N(0, 0.02)", "max_bs": 256,
             "n_rows": n_rows, "n_slots": n_slots, "kv_pool_gb": round(eng.kv_bytes / 1e9, 1),
             "weights_gb": round(weights.nbytes / 1e9, 1),
             "l2": "inputs larger than L2 (weights and K/V many times L2), no flush"}
    return shape, weights, eng, (lambda warm=False, gen=1: work), workload, extra


def measure(C, eng, stream, dev, make_work, steps, warmup, is_trace, world, local):
    """Warm up, then time `steps` iterations (fixed batch) or whole traces
    (trace: `steps` complete runs), with an event after every iteration."""
    import torch
    import torch.distributed as dist
    work = make_work(warm=True) if is_trace else make_work()
    for _ in range(max(3, warmup)):
        if is_trace and work.done():
            work = make_work(warm=True)
        work.step()
    if is_trace:   # the timed traces start fresh, from their first arrival
        while not work.done():
            work.step()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local)
    recs, evs, step_ms, usage, xfer = [], [], [], [], []
    runs = [make_work(gen=i + 1) for i in range(steps)] if is_trace else [work]
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for w in runs:
        n = 0
        while (not w.done()) if is_trace else n < steps:
            t0 = time.perf_counter()
            rec = w.step()
            step_ms.append(1000.0 * (time.perf_counter() - t0))
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            evs.append(ev)
            h2d, d2h, _ = C.orca_last_transfer(eng.handle)
            xfer.append((h2d, d2h))
            usage.append(C.orca_kv_usage(eng.handle, w.loop.pool.arr, w.loop.pool.n))
            recs.append(rec)
            n += 1
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - w0
    clocks = sampler.stop()
    it_ms = []
    prev = ev0
    for ev in evs:
        it_ms.append(prev.elapsed_time(ev))
        prev = ev
    return {"recs": recs, "it_ms": it_ms, "dev_s": sum(it_ms) / 1000.0, "wall": wall, "clocks": clocks,
            "step_ms": step_ms, "usage": usage, "xfer": xfer, "work": work}


def steady_state(recs, it_ms):
    """CS349D Lecture 2, results of section 5 (steady-state throughput): count
    only up to the iteration in which the last request produces its first
    token; after it the batch drains."""
    first = {}
    for k, rec in enumerate(recs):
        for rid, t in zip(rec.req_ids, rec.next_tokens):
            if t >= 0 and rid not in first:
                first[rid] = k
    end = max(first.values()) if first else len(recs) - 1
    s = sum(it_ms[:end + 1]) / 1000.0
    rows = sum(sum(r.n_new) for r in recs[:end + 1])
    gen = sum(sum(1 for t in r.next_tokens if t >= 0) for r in recs[:end + 1])
    done = sum(len(r.released) for r in recs[:end + 1])
    return {"iterations": end + 1, "seconds": s, "processed_tokens_per_s": rows / s, "generated_tokens_per_s": gen / s,
            "completed_requests_per_s": done / s,
            "window": "from the first iteration to the one in which the last request produced its first token"}


def run_config(args, config, rank, world, local, dev, stream):
    """Measure one workload; returns the JSON line (before printing)."""
    import torch
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import replicas
    from iteration_level_selective_gb300 import runtime as rt
    is_trace = config in TRACES
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[config]
    if is_trace:
        shape, trace_fn, max_bs, n_slots, max_rows, workload = trace_spec(config)
        if args.kv_slots:
            n_slots = args.kv_slots
        if args.reserve == "paged":
            n_slots -= n_slots % C.ORCA_KV_BLOCK   # whole K/V blocks
        host_w = synth.make_weights(shape, seed=0) if shape.n_layers * shape.hidden <= 12 * 768 else None
        weights = rt.DeviceWeights(shape, dev, host=host_w, seed=0)
        del host_w
        eng = rt.Engine(shape, weights, max_bs=max_bs, n_slots=n_slots, max_rows=max_rows, device=dev,
                        reserve_policy=rt.RESERVE_POLICIES[args.reserve])
        n_warm = [0]

        def make_work(warm=False, gen=1):
            """Timed trace number `gen` (1, 2, ...), or a short warm-up trace:
            the first 32 requests of another stream, at once, at most 8 tokens each."""
            if warm:
                n_warm[0] += 1
                trace = [synth.Request(r.req_id, 0, r.prompt, min(r.out_len, 8), r.max_tokens)
                         for r in trace_fn(rank, 10_000 + n_warm[0])[:32]]
            else:
                trace = trace_fn(rank, gen)
            return TraceWorkload(eng, trace, stream, args.token_budget or None, args.chunk or None, args.workers)
        extra = {"model": f"{'gpt2-small' if shape is synth.GPT2_SMALL else '13B'}-shaped, random init N(0, 0.02)",
                 "max_bs": max_bs, "n_slots": n_slots, "kv_pool_gb": round(eng.kv_bytes / 1e9, 1),
                 "l2": "inputs larger than L2 (weights + K/V pool), no flush",
                 "timed": f"{steps} complete trace(s) after a warm-up trace"}
        if args.token_budget or args.chunk:
            workload += f", chunked prefill (token budget {args.token_budget or 'none'}, chunk {args.chunk or 'none'})"
            extra["token_budget"], extra["chunk"] = args.token_budget or None, args.chunk or None
        if args.workers != 1:
            workload += f", {args.workers} batches in flight"
            extra["n_workers"] = args.workers
        if args.reserve != "max":
            workload += f", {args.reserve} K/V reservation"
            extra["reserve_policy"] = args.reserve
    else:
        shape, weights, eng, make_work, workload, extra = build_fixed(config, dev, stream)

    m = measure(C, eng, stream, dev, make_work, steps, args.warmup, is_trace, world, local)
    recs = m["recs"]
    n_it = len(recs)
    rows = sum(sum(r.n_new) for r in recs)
    gen_tok = sum(sum(1 for t in r.next_tokens if t >= 0) for r in recs)
    done = sum(len(r.released) for r in recs)
    launches = sum(r.launches for r in recs)
    h2d = sum(x[0] for x in m["xfer"])
    d2h = sum(x[1] for x in m["xfer"])
    (dev_s, wall), (rows, gen_tok, done, h2d, d2h, launches, n_it_all) = replicas.reduce_timing(
        [m["dev_s"], m["wall"]], [rows, gen_tok, done, h2d, d2h, launches, n_it], device=dev)

    def kernel_pass(mode):
        """The timed iterations again (the first timed trace, whole), with
        per-kernel-class timing: mode 2 = launch stamps in the graph-replayed
        forward, mode 1 = CUDA events around eagerly launched kernels."""
        C.orca_profile_enable(eng.handle, mode)
        t = time.perf_counter()
        if is_trace:
            pw, n = make_work(gen=1), 0
            while not pw.done():
                pw.step()
                n += 1
        else:
            pw, n = m["work"], n_it
            for _ in range(n_it):
                pw.step()
        torch.cuda.synchronize(dev)
        t = time.perf_counter() - t
        agg = kernel_classes(C, eng)
        C.orca_profile_enable(eng.handle, 0)
        return agg, n, t

    agg, n_prof, t_prof = kernel_pass(2)
    agg_ev, n_ev, t_ev = kernel_pass(1)
    peaks, peak_src = load_peaks()
    total_ms = sum(a["ms"] for a in agg.values()) or 1.0
    dom = max(agg, key=lambda k: agg[k]["ms"])
    batches = [list(zip(r.n_new, r.n_ctx)) for r in recs]
    it_roof = iteration_roofline(shape, float(weights.nbytes), batches, m["dev_s"], peaks)
    value = rows / dev_s
    config_obj = {"workload": workload}
    config_obj.update(extra)
    config_obj["parallelism"] = f"replicas x{world}"
    usage = m["usage"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n_it,
        "warmup": max(3, args.warmup), "ms_per_step": 1000.0 * dev_s / max(1, n_it),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_obj,
        "generated_tokens_per_s": gen_tok / dev_s,
        "completed_requests_per_s": done / dev_s,
        "e2e": {"value": rows / wall, "unit": UNIT, "h2d_bytes_per_step": h2d / n_it_all,
                "d2h_bytes_per_step": d2h / n_it_all},
        "gpu_launches": launches,
        "roofline": roofline_of(agg, dom, peaks, peak_src, config),
        "iteration_roofline": it_roof,
        "kernel_roofline": per_kernel_roofline(agg, peaks),
        "kernel_time_share": {k: round(v["ms"] / total_ms, 4) for k, v in agg.items()},
        "kernel_ms_per_step": {k: round(v["ms"] / max(1, n_prof), 4) for k, v in agg.items()},
        "kernel_timing": {
            "how": "the timed iterations again on the same path (graph replay); every kernel raises a %globaltimer "
                   "end stamp, a launch's share is its end minus the previous launch's end, so the classes add up "
                   "to each iteration's device time",
            "iterations": n_prof, "ms_per_step_wall": round(1000 * t_prof / max(1, n_prof), 4),
            "kernel_ms_sum_per_step": round(total_ms / max(1, n_prof), 4)},
        "event_pass": {
            "how": "the same iterations launched eagerly with a CUDA event pair around every kernel on the "
                   "iteration stream (no graph, no overlap between kernels)",
            "iterations": n_ev, "ms_per_step_wall": round(1000 * t_ev / max(1, n_ev), 4),
            "kernel_ms_per_step": {k: round(v["ms"] / max(1, n_ev), 4) for k, v in agg_ev.items()},
            "roofline_frac": {k: v.get("frac_tensor", v.get("frac_hbm")) for k, v in
                              per_kernel_roofline(agg_ev, load_peaks()[0]).items()}},
        "kv_usage": {"reserved_frac": round(float(np.mean([u[0] for u in usage])) / eng.cfg.n_slots, 5),
                     "stored_frac": round(float(np.mean([u[1] for u in usage])) / eng.cfg.n_slots, 5),
                     "stored_over_reserved": round(float(np.sum([u[1] for u in usage]) /
                                                         max(1, np.sum([u[0] for u in usage]))), 4),
                     "weighting": "per iteration, after each timed iteration"},
        "iteration_ms": {"p50": round(float(np.percentile(m["it_ms"], 50)), 4),
                         "p99": round(float(np.percentile(m["it_ms"], 99)), 4), "max": round(max(m["it_ms"]), 4),
                         "clock": "CUDA events between consecutive iterations on the iteration stream"},
        "clocks": m["clocks"],
    }
    if is_trace:
        line["steady_state"] = steady_state(recs, m["it_ms"])
        line["overall"] = {"processed_tokens_per_s": value, "generated_tokens_per_s": gen_tok / dev_s,
                           "completed_requests_per_s": done / dev_s, "iterations": n_it}
    if config == "13b-decode" or (not is_trace and "attention" in agg and config == "13b-mixed"):
        line["attention_roofline"] = roofline_of(agg, "attention", peaks, peak_src, config)
    _free_engine(eng, weights)
    return line


SUB_KEYS = ("value", "unit", "steps", "ms_per_step", "config", "roofline", "attention_roofline", "kernel_timing",
            "event_pass", "iteration_roofline", "kernel_roofline", "kernel_ms_per_step", "gpu_launches", "e2e", "clocks",
            "steady_state", "overall", "completed_requests_per_s", "generated_tokens_per_s")


def run_ours(args, rank: int, world: int):
    import torch
    from iteration_level_selective_gb300 import build as B

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    stream = torch.cuda.Stream(dev)
    line = run_config(args, args.config, rank, world, local, dev, stream)
    if args.config == "13b-mixed" and not args.no_sub:
        # the decode-dominated iteration, for the attention kernel's HBM target
        sub_args = argparse.Namespace(**vars(args))
        sub_args.steps = None
        sub = run_config(sub_args, "13b-decode", rank, world, local, dev, stream)
        line["decode_stress"] = {k: sub[k] for k in SUB_KEYS if k in sub}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc = cpu_oracle_sample(args.config, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed iterations (13b-mixed: 10, 13b-decode: 50); trace workloads: complete traces (1)")
    ap.add_argument("--config", choices=CONFIGS, default=DEFAULT_CONFIG,
                    help="13b-mixed (default: the prefill-heavy 13B iteration, with the decode-stress iteration as "
                         "a sub-result), 13b-decode, 13b-trace (the 13B serving trace), gpt2-trace")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sub", action="store_true", help="13b-mixed: skip the decode-stress sub-result")
    ap.add_argument("--token-budget", type=int, default=0,
                    help="trace workloads: chunked prefill with this many rows per iteration at most")
    ap.add_argument("--chunk", type=int, default=0, help="trace workloads: prompt chunk size for chunked prefill")
    ap.add_argument("--workers", type=int, choices=[1, 2], default=1,
                    help="trace workloads: batches in flight at once (Algorithm 1's n_workers)")
    ap.add_argument("--reserve", choices=["max", "pow2", "oracle", "paged"], default="max",
                    help="trace workloads: K/V reservation policy (max_tokens, power of two, true length) or paged "
                         "K/V (32-slot blocks on demand, preemption of the latest arrival)")
    ap.add_argument("--kv-slots", type=int, default=0,
                    help="trace workloads: K/V pool slots (default: 40 GB worth for gpt2-trace, 120 GB for 13b-trace)")
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

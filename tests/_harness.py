"""Shared helpers of the parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare."""
import numpy as np

import synth
from oracle import model as omodel
from oracle import scheduler as osched


def max_rel_err(got, want):
    """max_j |g_j - o_j| / max_j |o_j| over one logits row."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.abs(got - want).max() / np.abs(want).max())


def run_gpu(shape, host_weights, trace, max_bs, n_slots, max_rows, teacher_force=False, keep_ids=None,
            keep_all=False, eager=False, token_budget=None, chunk=None, reserve_policy=0, n_workers=1):
    import torch
    from iteration_level_selective_gb300 import runtime as rt
    dev = torch.device("cuda:0")
    w = rt.DeviceWeights(shape, dev, host=host_weights)
    eng = rt.Engine(shape, w, max_bs=max_bs, n_slots=n_slots, max_rows=max_rows, device=dev,
                    reserve_policy=reserve_policy)
    pool = rt.RequestPool(trace, teacher_force=teacher_force)
    loop = rt.ServingLoop(eng, pool, teacher_force=teacher_force, keep_logits=keep_all, keep_ids=keep_ids,
                          eager=eager, token_budget=token_budget, chunk=chunk, n_workers=n_workers, track_kv=True)
    recs = loop.run()
    return recs, eng, pool


def compare_schedule(gpu_recs, trace, max_bs, n_slots, token_budget=None, chunk=None, reserve_policy=0,
                     n_workers=1):
    """Integer record of every iteration, bit-exact against the oracle scheduler."""
    orecs = osched.run_schedule(trace, max_bs=max_bs, n_slots=n_slots, token_budget=token_budget, chunk=chunk,
                                policy=reserve_policy, n_workers=n_workers)
    assert len(gpu_recs) == len(orecs)
    for g, o in zip(gpu_recs, orecs):
        assert (g.it, g.req_ids, g.n_new, g.n_ctx, g.slot_base, sorted(g.released), sorted(g.preempted)) == \
               (o.it, o.req_ids, o.n_new, o.n_ctx, o.slot_base, sorted(o.released), sorted(o.preempted)), (g, o)
        if g.kv is not None:   # reserved and stored K/V slots after the iteration
            assert tuple(g.kv) == tuple(o.kv), (g.it, g.kv, o.kv)
    return orecs


def gpu_logits_by_request(recs):
    """request id -> list of logits rows in generation order (iterations
    that ran a prompt chunk without completing the prompt generate nothing
    and are skipped)."""
    out = {}
    for rec in recs:
        if rec.logits is None:
            continue
        emitted = {rid for rid, t in zip(rec.req_ids, rec.next_tokens) if t >= 0}
        if isinstance(rec.logits, dict):
            for rid, row in rec.logits.items():
                if rid in emitted:
                    out.setdefault(rid, []).append(row)
        else:
            for k, rid in enumerate(rec.req_ids):
                if rid in emitted:
                    out.setdefault(rid, []).append(rec.logits[k])
    return out


def gpu_tokens_by_request(recs):
    out = {}
    for rec in recs:
        for rid, t in zip(rec.req_ids, rec.next_tokens):
            if t >= 0:
                out.setdefault(rid, []).append(t)
    return out


def oracle_generate(shape, host_weights, req, teacher_force, stop_after=None):
    orc = omodel.GPTOracle(shape, host_weights)
    greedy, logits, _ = orc.generate(req.prompt, req.out_len, forced=req.forced if teacher_force else None,
                                     stop_after=stop_after)
    return greedy, logits


def n_generated(req):
    return min(req.out_len, req.max_tokens - req.n_prompt)

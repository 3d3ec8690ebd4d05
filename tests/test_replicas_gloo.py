"""Replica path on CPU: two gloo ranks, each driving its own host-only
engine (scheduler + slot pool) over its own trace; the timing reduction
takes the slowest rank and sums the work."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    import ctypes
    import numpy as np
    import torch.distributed as dist
    import synth
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import replicas
    from oracle import scheduler as osched

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    trace = synth.make_trace(20, (1, 30), (1, 20), vocab=100, seed=replicas.trace_seed(rank), rate_per_iter=0.8)
    cfg = C.orca_config(n_layers=1, hidden=64, n_heads=4, ffn=256, vocab=100, max_pos=64, dtype=0, max_bs=4,
                        n_slots=120, max_rows=128)
    eng = C.orca_engine_create(cfg)
    reqs = sorted(trace, key=lambda r: (r.arrival, r.req_id))
    arr = (C.orca_request * len(reqs))()
    bufs = []
    for i, r in enumerate(reqs):
        b = np.zeros(r.n_prompt + r.out_len, dtype=np.int32)
        bufs.append(b)
        arr[i] = C.orca_request(req_id=r.req_id, arrival=r.arrival, state=0, n_prompt=r.n_prompt,
                                max_tokens=r.max_tokens, out_len=r.out_len, n_cached=0, n_generated=0, slot_base=-1,
                                tokens=b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    bi = (ctypes.c_int32 * 4)()
    it, n_arr, done, rows = 0, 0, 0, 0
    while done < len(reqs):
        if n_arr == done and reqs[n_arr].arrival > it:
            it = reqs[n_arr].arrival
        while n_arr < len(reqs) and reqs[n_arr].arrival <= it:
            n_arr += 1
        nb = C.orca_select_batch(eng, arr, n_arr, bi)
        for k in range(nb):   # host-only engine: apply the post-iteration update here
            a = arr[bi[k]]
            L = a.n_prompt - a.n_cached if a.n_cached < a.n_prompt else 1
            rows += L
            a.state, a.n_cached, a.n_generated = 1, a.n_cached + L, a.n_generated + 1
            if a.n_generated >= a.out_len or a.n_prompt + a.n_generated >= a.max_tokens:
                a.state = 3
                C.orca_kv_release(eng, a.req_id)
                done += 1
        it += 1
    C.orca_engine_destroy(eng)
    want_rows = sum(sum(r.n_new) for r in osched.run_schedule(trace, max_bs=4, n_slots=120))
    assert rows == want_rows
    secs, counts = replicas.reduce_timing([0.5 + rank, 1.0], [rows, 1])
    dist.barrier()
    out[rank] = (rows, secs, counts)
    dist.destroy_process_group()


def test_two_gloo_replicas_reduce_max_time_and_sum_work(liborca):
    mp = torch.multiprocessing.get_context("spawn")
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    procs = [mp.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    rows0, secs0, counts0 = out[0]
    rows1, secs1, counts1 = out[1]
    assert rows0 != rows1                      # independent request streams
    assert secs0 == secs1 == [1.5, 1.0]        # slowest rank
    assert counts0 == counts1 == [rows0 + rows1, 2]

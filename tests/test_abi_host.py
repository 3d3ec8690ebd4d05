"""C-ABI checks that need no GPU: exported symbols, host-only engine,
Algorithm 1 Select and the slot pool, bit-exact against the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

from iteration_level_selective_gb300 import _orca as C
from oracle import scheduler as osched

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "orca.h")


def _declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^int\s+(orca_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(liborca):
    names = _declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(liborca, n), n
    assert set(names) <= set(C.EXPORTS) | set(names)
    assert set(C.EXPORTS) <= set(names)


def _cfg(max_bs=4, n_slots=64, dtype=C.ORCA_DTYPE_F32, policy=C.ORCA_RESERVE_MAX):
    return C.orca_config(n_layers=2, hidden=64, n_heads=4, ffn=256, vocab=256, max_pos=64, dtype=dtype,
                         max_bs=max_bs, n_slots=n_slots, max_rows=64, reserve_policy=policy)


def test_sizes_and_config_validation(liborca):
    cfg = _cfg()
    assert C.orca_kv_pool_bytes(cfg) == 2 * 2 * 64 * 64 * 4
    assert C.orca_weight_count(cfg) == 4 + 12 * 2
    assert C.orca_workspace_bytes(cfg) > 0
    bad = _cfg()
    bad.n_heads = 3
    with pytest.raises(C.OrcaError):
        C.orca_workspace_bytes(bad)
    bad = _cfg(dtype=C.ORCA_DTYPE_BF16)   # hidden 64 ok, ffn 256 ok
    C.orca_workspace_bytes(bad)
    bad.hidden, bad.n_heads = 96, 6        # bf16 needs hidden % 64 == 0
    with pytest.raises(C.OrcaError):
        C.orca_workspace_bytes(bad)


def test_host_only_engine_reserve_release_errors(liborca):
    eng = C.orca_engine_create(_cfg(n_slots=20))
    try:
        assert [C.orca_kv_reserve(eng, i, 5) for i in range(3)] == [0, 5, 10]
        C.orca_kv_release(eng, 1)
        with pytest.raises(C.OrcaError) as ei:
            C.orca_kv_reserve(eng, 3, 6)        # 16 <= 20 but no hole of 6
        assert ei.value.code == C.ORCA_ENOSLOTS
        assert C.orca_kv_stats(eng) == (10, 2, 1)
        assert C.orca_kv_reserve(eng, 4, 5) == 5
        with pytest.raises(C.OrcaError) as ei:
            C.orca_kv_release(eng, 1)
        assert ei.value.code == C.ORCA_EDOUBLE_RELEASE
        with pytest.raises(C.OrcaError) as ei:
            C.orca_kv_release(eng, 99)
        assert ei.value.code == C.ORCA_EUNKNOWN_REQ
        with pytest.raises(C.OrcaError) as ei:
            C.orca_kv_reserve(eng, 0, 1)        # already holds a reservation
        assert ei.value.code == C.ORCA_EINVAL
        with pytest.raises(C.OrcaError) as ei:
            C.orca_kv_reserve(eng, 7, 0)
        assert ei.value.code == C.ORCA_EINVAL
        # profiling modes: 0 off, 1 events, 2 launch stamps; a host-only engine profiles nothing
        C.orca_profile_enable(eng, 0)
        for mode, code in ((3, C.ORCA_EINVAL), (-1, C.ORCA_EINVAL), (1, C.ORCA_ESTATE), (2, C.ORCA_ESTATE)):
            with pytest.raises(C.OrcaError) as ei:
                C.orca_profile_enable(eng, mode)
            assert ei.value.code == code, mode
        # orca_iteration needs a device side
        pool = (C.orca_request * 1)()
        bi = (ctypes.c_int32 * 4)()
        nt = (ctypes.c_int32 * 4)()
        with pytest.raises(C.OrcaError) as ei:
            C.orca_iteration(eng, pool, bi, 1, 0, nt)
        assert ei.value.code == C.ORCA_ESTATE
        with pytest.raises(C.OrcaError) as ei:
            C.orca_iteration_submit(eng, pool, bi, 1, 0)
        assert ei.value.code == C.ORCA_ESTATE
        with pytest.raises(C.OrcaError) as ei:
            C.orca_iteration_wait(eng, bi, nt)
        assert ei.value.code == C.ORCA_ESTATE
    finally:
        C.orca_engine_destroy(eng)


class _Sim:
    """Drives the C Select and the oracle Select side by side; the test
    applies the same post-iteration update to both."""

    def __init__(self, trace, max_bs, n_slots, budget=None, policy=C.ORCA_RESERVE_MAX):
        self.budget = budget  # (token_budget, chunk) for the chunked-prefill Select, or None
        self.policy = policy
        self.trace = sorted(trace, key=lambda t: (t[1], t[0]))
        self.eng = C.orca_engine_create(_cfg(max_bs=max_bs, n_slots=n_slots, policy=policy))
        self.max_bs = max_bs
        n = len(self.trace)
        self.arr = (C.orca_request * n)()
        self.bufs = []
        for i, (rid, arrival, lp, lo, mt) in enumerate(self.trace):
            b = np.zeros(lp + lo, dtype=np.int32)
            self.bufs.append(b)
            self.arr[i] = C.orca_request(req_id=rid, arrival=arrival, state=C.ORCA_INITIATION, n_prompt=lp,
                                         max_tokens=mt, out_len=lo, n_cached=0, n_generated=0, slot_base=-1,
                                         tokens=b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
        self.ostates = [osched.ReqState(rid, a, lp, lo, mt) for rid, a, lp, lo, mt in self.trace]
        self.oslots = osched.BlockPool(n_slots) if policy == C.ORCA_RESERVE_PAGED else osched.SlotPool(n_slots)
        self.bi = (ctypes.c_int32 * max_bs)()

    def run(self):
        it, n_arr, done = 0, 0, 0
        n = len(self.trace)
        while done < n:
            if n_arr == done and self.trace[n_arr][1] > it:
                it = self.trace[n_arr][1]
            while n_arr < n and self.trace[n_arr][1] <= it:
                n_arr += 1
            opool = [s for s in self.ostates[:n_arr] if s.state != osched.FINISHED]
            if self.budget is None:
                nb = C.orca_select_batch(self.eng, self.arr, n_arr, self.bi)
                osel = [(r, osched.default_rows(r))
                        for r in osched.select(opool, self.oslots, self.max_bs, self.policy)]
            else:
                nb = C.orca_select_batch_budget(self.eng, self.arr, n_arr, self.budget[0], self.budget[1], self.bi)
                osel = osched.select_budget(opool, self.oslots, self.max_bs, *self.budget, policy=self.policy)
            orun = [(r, k) for r, k in osel if k > 0]
            got = [(self.arr[self.bi[i]].req_id, self.arr[self.bi[i]].slot_base, self.arr[self.bi[i]].n_sched)
                   for i in range(nb)]
            want = [(r.req_id, r.slot_base, k) for r, k in orun]
            assert got == want, (it, got, want)
            assert C.orca_kv_stats(self.eng)[0] == self.oslots.n_rsrv
            assert C.orca_kv_usage(self.eng, self.arr, n_arr) == osched.kv_usage(self.ostates[:n_arr], self.oslots)
            for i in range(nb):
                a = self.arr[self.bi[i]]
                assert a.state == C.ORCA_RUNNING
                L = a.n_sched
                a.state, a.n_sched, a.n_cached = C.ORCA_INCREMENT, 0, a.n_cached + L
                if a.n_cached < a.n_prompt + a.n_generated:
                    continue
                a.n_generated += 1
                if a.n_generated >= a.out_len or a.n_prompt + a.n_generated >= a.max_tokens:
                    a.state = C.ORCA_FINISHED
                    C.orca_kv_release(self.eng, a.req_id)
                    done += 1
            for r, k in osel:
                r.state = osched.INCREMENT
                if k == 0:
                    continue
                r.n_cached += k
                if r.n_cached < osched.known_len(r):
                    continue
                r.n_generated += 1
                if osched.finished(r):
                    r.state = osched.FINISHED
                    self.oslots.release(r.req_id)
            # requests admitted without a row wait in INCREMENT, preempted ones in
            # INITIATION, on both sides
            for j in range(n_arr):
                if self.arr[j].state in (C.ORCA_INCREMENT, C.ORCA_INITIATION):
                    assert self.arr[j].state == self.ostates[j].state, (it, j)
                    assert self.arr[j].n_cached == self.ostates[j].n_cached
            it += 1
        C.orca_engine_destroy(self.eng)
        return it


def test_select_bit_exact_vs_oracle_random_traces(liborca):
    rng = np.random.default_rng(21)
    for trial in range(40):
        n = int(rng.integers(3, 60))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 20)), int(rng.integers(1, 25))
            trace.append((int(rng.permutation(1000)[i] if trial % 2 else i), int(rng.integers(0, 30)), lp, lo,
                          lp + lo + int(rng.integers(0, 8))))
        max_t = max(t[4] for t in trace)
        _Sim(trace, max_bs=int(rng.integers(1, 12)), n_slots=int(rng.integers(max_t, 4 * max_t))).run()


def test_budget_select_bit_exact_vs_oracle_random_traces(liborca):
    rng = np.random.default_rng(22)
    for trial in range(40):
        n = int(rng.integers(3, 40))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 40)), int(rng.integers(1, 12))
            trace.append((i, int(rng.integers(0, 30)), lp, lo, lp + lo + int(rng.integers(0, 8))))
        max_t = max(t[4] for t in trace)
        budget = (int(rng.integers(1, 48)), int(rng.integers(1, 32)))
        _Sim(trace, max_bs=int(rng.integers(1, 12)), n_slots=int(rng.integers(max_t, 4 * max_t)), budget=budget).run()


@pytest.mark.parametrize("policy", [C.ORCA_RESERVE_POW2, C.ORCA_RESERVE_ORACLE])
def test_reserve_policy_select_bit_exact_vs_oracle(liborca, policy):
    rng = np.random.default_rng(23 + policy)
    for trial in range(30):
        n = int(rng.integers(3, 40))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 30)), int(rng.integers(1, 20))
            trace.append((i, int(rng.integers(0, 30)), lp, lo, lp + lo + int(rng.integers(0, 30))))
        max_t = max(t[4] for t in trace)
        budget = (int(rng.integers(1, 48)), int(rng.integers(1, 32))) if trial % 2 else None
        _Sim(trace, max_bs=int(rng.integers(1, 12)), n_slots=int(rng.integers(max_t, 3 * max_t)), budget=budget,
             policy=policy).run()


def test_paged_select_bit_exact_vs_oracle(liborca):
    rng = np.random.default_rng(26)
    for trial in range(30):
        n = int(rng.integers(2, 25))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 60)), int(rng.integers(1, 30))
            trace.append((i, int(rng.integers(0, 20)), lp, lo, lp + lo + int(rng.integers(0, 4))))
        need = max(-(-(t[2] + t[3]) // 32) for t in trace)
        budget = (int(rng.integers(8, 64)), int(rng.integers(4, 40))) if trial % 2 else None
        _Sim(trace, max_bs=int(rng.integers(1, 9)), n_slots=32 * int(rng.integers(need, 2 * need + 2)),
             budget=budget, policy=C.ORCA_RESERVE_PAGED).run()


def test_paged_engine_has_no_reservations(liborca):
    eng = C.orca_engine_create(_cfg(n_slots=64, policy=C.ORCA_RESERVE_PAGED))
    try:
        with pytest.raises(C.OrcaError) as ei:
            C.orca_kv_reserve(eng, 1, 4)
        assert ei.value.code == C.ORCA_ESTATE
    finally:
        C.orca_engine_destroy(eng)


def test_bad_reserve_policy_rejected(liborca):
    with pytest.raises(C.OrcaError) as ei:
        C.orca_kv_pool_bytes(_cfg(policy=4))
    assert ei.value.code == C.ORCA_EINVAL
    with pytest.raises(C.OrcaError) as ei:   # paged K/V: whole blocks
        C.orca_kv_pool_bytes(_cfg(n_slots=100, policy=C.ORCA_RESERVE_PAGED))
    assert ei.value.code == C.ORCA_EINVAL


def test_budget_select_rejects_bad_budget(liborca):
    eng = C.orca_engine_create(_cfg(max_bs=4, n_slots=100))
    try:
        pool = (C.orca_request * 1)()
        bi = (ctypes.c_int32 * 4)()
        for tb, ch in ((0, 4), (4, 0), (-1, 4)):
            with pytest.raises(C.OrcaError) as ei:
                C.orca_select_batch_budget(eng, pool, 0, tb, ch, bi)
            assert ei.value.code == C.ORCA_EINVAL
    finally:
        C.orca_engine_destroy(eng)


def test_select_break_no_skip_via_abi(liborca):
    # head does not fit: later smaller requests are not admitted
    sim = _Sim([(0, 0, 2, 5, 8), (1, 1, 2, 2, 4), (2, 2, 1, 1, 2)], max_bs=8, n_slots=10)
    n_iters = sim.run()
    assert n_iters == 5 + 2   # request 0 alone for 5 iterations, then 1 and 2 together


def test_select_rejects_bad_request(liborca):
    eng = C.orca_engine_create(_cfg())
    arr = (C.orca_request * 1)()
    b = np.zeros(4, dtype=np.int32)
    arr[0] = C.orca_request(req_id=1, arrival=0, state=C.ORCA_INITIATION, n_prompt=3, max_tokens=2, out_len=1,
                            n_cached=0, n_generated=0, slot_base=-1,
                            tokens=b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    bi = (ctypes.c_int32 * 4)()
    with pytest.raises(C.OrcaError):
        C.orca_select_batch(eng, arr, 1, bi)
    C.orca_engine_destroy(eng)

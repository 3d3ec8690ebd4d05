"""The device-side failure path and buffer bounds, on the GPU, with no fault.

Every wait inside the kernels is bounded: a self-test kernel waits on a
barrier that nothing completes, and the test checks that the wait expires,
raises the status word and leaves the context usable.  Guard bands around
the K/V pool and the workspace check that no kernel of a whole serving run
writes outside the buffers it is given.
"""
import time

import numpy as np
import pytest

import synth

from . import _harness as hz

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL_BF16 = synth.ModelShape(n_layers=2, hidden=256, n_heads=4, ffn=1024, vocab=1000, max_pos=1024,
                              dtype=synth.DTYPE_BF16)


@pytest.fixture(scope="module")
def cuda(liborca):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def test_bounded_wait_expires_and_the_context_survives(cuda):
    from iteration_level_selective_gb300 import _orca as C
    st = torch.cuda.current_stream()
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    C.orca_selftest_wait_timeout(status.data_ptr(), st.cuda_stream)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == 1, int(status.item())   # wait timeout, nothing else
    assert 1.0 < waited < 30.0, waited                     # the bound, not an immediate return
    # kernels still run and are right afterwards: one Linear against fp64
    rng = np.random.default_rng(3)
    M, N, K = 64, 256, 128
    A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy((rng.standard_normal((N, K)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    ref = A.double() @ W.double().T
    out = torch.zeros((M, N), dtype=torch.float32, device=cuda)
    status.zero_()
    Ad, Wd = A.to(cuda), W.to(cuda)
    C.orca_linear(C.ORCA_DTYPE_BF16, C.ORCA_LINEAR_F32OUT, Ad.data_ptr(), Wd.data_ptr(), 0, out.data_ptr(), M, N,
                  K, status.data_ptr(), st.cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    err = (out.double().cpu() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err


class _GuardedEngine:
    """An engine whose K/V pool and workspace sit between guard bands of a
    known byte pattern (the same attributes ServingLoop reads from
    runtime.Engine)."""

    GUARD = 1 << 20   # bytes on each side; a multiple of 256 keeps the alignment
    PATTERN = 0xA5

    def __init__(self, shape, weights, max_bs, n_slots, max_rows, device, reserve_policy):
        from iteration_level_selective_gb300 import _orca as C
        from iteration_level_selective_gb300 import runtime as rt
        self.shape, self.device, self.max_bs = shape, device, max_bs
        self.cfg = rt.make_config(shape, max_bs, n_slots, max_rows, reserve_policy)
        self.kv_bytes = C.orca_kv_pool_bytes(self.cfg)
        self.ws_bytes = C.orca_workspace_bytes(self.cfg)
        G = self.GUARD
        self.kv_all = torch.full((self.kv_bytes + 2 * G,), self.PATTERN, dtype=torch.uint8, device=device)
        self.ws_all = torch.full((self.ws_bytes + 2 * G,), self.PATTERN, dtype=torch.uint8, device=device)
        self.weights = weights
        self.handle = C.orca_engine_create(self.cfg, weights.ptrs, self.kv_all.data_ptr() + G, self.kv_bytes,
                                           self.ws_all.data_ptr() + G, self.ws_bytes)

    def guards_intact(self):
        G, p = self.GUARD, self.PATTERN
        torch.cuda.synchronize()
        return {name: bool((buf[:G] == p).all().item() and (buf[G + n:] == p).all().item())
                for name, buf, n in (("kv", self.kv_all, self.kv_bytes), ("workspace", self.ws_all, self.ws_bytes))}

    def close(self):
        from iteration_level_selective_gb300 import _orca as C
        if self.handle:
            C.orca_engine_destroy(self.handle)
            self.handle = None


@pytest.mark.parametrize("policy", ["max", "paged"])
def test_no_kernel_writes_outside_its_buffers(cuda, policy):
    """A bf16 trace with prompts on both attention kernels, decodes, releases
    and (paged) preemption; afterwards every guard byte is unchanged."""
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import runtime as rt
    shape = SMALL_BF16
    w = synth.make_weights(shape, seed=23, w_std=0.05, bias_std=0.02, ln_std=0.1)
    # prompts up to 160 tokens fit the 192-slot paged pool (6 blocks of 32) one at a time
    trace = synth.make_trace(10, (1, 160), (10, 60), vocab=shape.vocab, seed=24, rate_per_iter=1.5, forced=True)
    pol = C.ORCA_RESERVE_PAGED if policy == "paged" else C.ORCA_RESERVE_MAX
    n_slots = 6 * 32 if policy == "paged" else 4000
    dw = rt.DeviceWeights(shape, cuda, host=w)
    eng = _GuardedEngine(shape, dw, max_bs=6, n_slots=n_slots, max_rows=2048, device=cuda, reserve_policy=pol)
    try:
        pool = rt.RequestPool(trace, teacher_force=True)
        loop = rt.ServingLoop(eng, pool, teacher_force=True, keep_logits=True)
        recs = loop.run()
        assert loop.done() and len(recs) > 0
        assert eng.guards_intact() == {"kv": True, "workspace": True}
        # and the run itself was right: logits of every request within the bf16 bound
        got = hz.gpu_logits_by_request(recs)
        for req in trace[:4]:
            _, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
            for g, o in zip(got[req.req_id], logits):
                assert hz.max_rel_err(g, o) < 2e-2
    finally:
        eng.close()


def test_iteration_reports_an_expired_wait_and_the_engine_goes_on(cuda):
    """An iteration whose status word a bounded wait raised (the self-test
    hook: one CTA waits on a barrier nothing completes) returns ORCA_EDEVICE
    after the bound; requests admitted afterwards on the same engine, and a
    fresh engine, still match the oracle."""
    import ctypes
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import runtime as rt
    shape = SMALL_BF16
    w = synth.make_weights(shape, seed=25, w_std=0.05, bias_std=0.02, ln_std=0.1)
    dw = rt.DeviceWeights(shape, cuda, host=w)
    eng = rt.Engine(shape, dw, max_bs=4, n_slots=2000, max_rows=512, device=cuda)
    try:
        bad = synth.make_trace(2, (40, 60), (3, 3), vocab=shape.vocab, seed=26, forced=True)
        pool = rt.RequestPool(bad, teacher_force=True)
        bi, nt = (ctypes.c_int32 * 4)(), (ctypes.c_int32 * 4)()
        nb = C.orca_select_batch(eng.handle, pool.arr, pool.n, bi)
        assert nb == 2
        t0 = time.perf_counter()
        with pytest.raises(C.OrcaError) as ei:
            C.orca_iteration(eng.handle, pool.arr, bi, nb, C.ORCA_ITER_TEACHER_FORCE | C.ORCA_ITER_SELFTEST_TIMEOUT,
                             nt)
        assert ei.value.code == C.ORCA_EDEVICE
        assert 1.0 < time.perf_counter() - t0 < 30.0
        # new requests on the same engine (the failed ones keep their slots)
        good = [synth.Request(100 + r.req_id, 0, r.prompt, r.out_len, r.max_tokens, forced=r.forced)
                for r in synth.make_trace(3, (1, 80), (2, 5), vocab=shape.vocab, seed=27, forced=True)]
        loop = rt.ServingLoop(eng, rt.RequestPool(good, teacher_force=True), teacher_force=True, keep_logits=True)
        got = hz.gpu_logits_by_request(loop.run())
        for req in good:
            _, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
            for g, o in zip(got[req.req_id], logits):
                assert hz.max_rel_err(g, o) < 2e-2
    finally:
        eng.close()
    # and a fresh engine serves the requests that failed
    recs, eng2, _ = hz.run_gpu(shape, w, bad, max_bs=4, n_slots=2000, max_rows=512, teacher_force=True,
                               keep_all=True)
    try:
        got = hz.gpu_logits_by_request(recs)
        for req in bad:
            _, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
            for g, o in zip(got[req.req_id], logits):
                assert hz.max_rel_err(g, o) < 2e-2
    finally:
        eng2.close()

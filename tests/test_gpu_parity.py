"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars (from the method's tolerance): integer work bit-exact (schedule,
reservations, releases, ragged descriptor, greedy tokens on forced logits);
logits within max relative error 1e-4 per row in fp32 models and 2e-2 in
bf16 models, under teacher forcing where the CUDA path's own greedy choice
could otherwise diverge from the oracle's.
"""
import numpy as np
import pytest

import synth
from oracle import scheduler as osched
from oracle import ragged as oragged

from . import _harness as hz

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FP32_TOL = 1e-4
BF16_TOL = 2e-2


@pytest.fixture(scope="module")
def cuda(liborca):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


# ------------------------------------------------------------------ kernels

def test_argmax_forced_logits_bit_exact(cuda):
    from iteration_level_selective_gb300 import _orca as C
    rng = np.random.default_rng(0)
    V = 50257
    lg = rng.standard_normal((37, V)).astype(np.float32)
    lg[3, [10, 500, 40000]] = 100.0                 # tie: lowest index wins
    lg[4, :] = 1.0                                  # all equal -> 0
    lg[5, 7] = np.nan                               # NaN never wins
    lg[5, 9] = 50.0
    lg[6, :] = -np.inf
    lg[6, V - 1] = -1e30
    want = np.argmax(np.where(np.isnan(lg), -np.inf, lg), axis=1)
    d = torch.from_numpy(lg).to(cuda)
    out = torch.full((37,), -7, dtype=torch.int32, device=cuda)
    C.orca_argmax_rows(d.data_ptr(), 37, V, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got, want)
    assert got[3] == 10 and got[4] == 0 and got[5] == 9 and got[6] == V - 1


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (300, 1000, 768), (257, 2304, 768), (2048, 3072, 768),
                                   (64, 50257, 768), (64, 768, 3072), (130, 2304, 768), (3000, 5120, 1024),
                                   (600, 2304, 768),
                                   # one row tile with all of K in flight at once (64- and 128-row A
                                   # boxes, a ragged last column tile, a single k stage)
                                   (64, 768, 768), (100, 768, 512), (17, 1000, 1024), (5, 3072, 256),
                                   # one row tile and a long K: split-K over a cluster (ragged N, 64- and
                                   # 128-row A boxes, uneven K ranges)
                                   (37, 300, 2048), (100, 768, 3072), (1, 1000, 4096), (128, 520, 2112),
                                   # few narrow tiles with a 1 MB weight block each: split-K over the
                                   # persistent kernel when a scratch buffer is given
                                   (200, 520, 16384),
                                   # CTA-pair kernel (256 x 256 tiles over two SMs, when its waves beat the
                                   # single CTA's): ragged last pair tile (one row in the leader, none in the
                                   # peer), a single k-block with ragged N, vocab-wide ragged N, a long K;
                                   # wide N and K on single CTAs (two waves against three)
                                   (513, 5120, 512), (1024, 20000, 64), (777, 50257, 1024), (300, 12288, 4096),
                                   (1500, 4096, 5120), (200, 15360, 512),
                                   # a weight stream of >= 128 MB at a few hundred rows: CTA-pair tiles
                                   # shared out along K when a scratch buffer is given (without one: whole
                                   # pair tiles, or 256-wide single-CTA tiles) - 2 and 3 equal k-ranges per
                                   # tile (ragged N and K), stream ranges over 79 tiles with 2 pieces a tile
                                   # (ragged N), over 40 tiles in two ragged rows with up to 3 pieces
                                   (200, 5120, 5120), (300, 4096, 16384), (200, 5000, 13440), (250, 20000, 4096),
                                   (300, 5000, 13440),
                                   # a very long K on three tiles: 25 pieces a tile, more than the ring's slots
                                   # (the last pair reads them back through registers)
                                   (200, 520, 131072)])
@pytest.mark.parametrize("mode", ["store", "gelu", "resid", "f32out"])
@pytest.mark.parametrize("split", [False, True])
def test_linear_bf16_tcgen05_vs_fp64(cuda, M, N, K, mode, split):
    from iteration_level_selective_gb300 import _orca as C
    if mode != "f32out" and N == 50257:
        pytest.skip("vocab-wide output only in fp32")
    rng = np.random.default_rng(M * 7 + N)
    A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy((rng.standard_normal((N, K)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    bias = torch.from_numpy(rng.standard_normal(N).astype(np.float32))
    ref = A.double() @ W.double().T + bias.double()
    x0 = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32))
    if mode == "gelu":
        ref = torch.nn.functional.gelu(ref, approximate="tanh")
    if mode == "resid":
        ref = ref + x0.double()
    Ad, Wd, bd = A.to(cuda), W.to(cuda), bias.to(cuda)
    if mode in ("store", "gelu"):
        out = torch.zeros((M, N), dtype=torch.bfloat16, device=cuda)
    else:
        out = (x0.clone() if mode == "resid" else torch.zeros((M, N))).to(cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    m = {"store": C.ORCA_LINEAR_STORE, "gelu": C.ORCA_LINEAR_GELU, "resid": C.ORCA_LINEAR_RESID,
         "f32out": C.ORCA_LINEAR_F32OUT}[mode]
    scratch = torch.empty(64 << 20, dtype=torch.uint8, device=cuda) if split else None
    C.orca_linear(C.ORCA_DTYPE_BF16, m, Ad.data_ptr(), Wd.data_ptr(), bd.data_ptr(), out.data_ptr(), M, N, K,
                  status.data_ptr(), torch.cuda.current_stream().cuda_stream,
                  scratch_ptr=scratch.data_ptr() if split else 0, scratch_bytes=(64 << 20) if split else 0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.double().cpu()
    scale = ref.abs().max().item()
    # fp32 accumulation of exact bf16 products (its rounding error grows with the K / 16 chained
    # MMAs: 1e-5 up to K = 4096, in proportion beyond); bf16 output rounding (2^-8) for store/gelu
    tol = 2 ** -7 if mode in ("store", "gelu") else 1e-5 * max(1.0, K / 4096)
    err = (got - ref).abs().max().item() / scale
    assert err < tol, err


@pytest.mark.parametrize("M,N,K", [(1, 50257, 768), (64, 50257, 768), (200, 1000, 256), (7, 300, 64),
                                   # CTA-pair tiles shared out along K in stream ranges
                                   (250, 20000, 4096)])
def test_fused_argmax_matches_argmax_of_stored_logits(cuda, M, N, K):
    """The LM head's fused greedy choice equals the argmax of the same
    call's fp32 logits, bit for bit (lowest index on ties)."""
    from iteration_level_selective_gb300 import _orca as C
    rng = np.random.default_rng(M + N)
    A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16).to(cuda)
    # a few duplicated weight rows create exact ties between columns
    Wn = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    Wn[N // 2] = Wn[N // 3]
    W = torch.from_numpy(Wn).to(torch.bfloat16).to(cuda)
    out = torch.empty((M, N), dtype=torch.float32, device=cuda)
    keys = torch.full((M,), -1, dtype=torch.int64, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    scratch = torch.empty(64 << 20, dtype=torch.uint8, device=cuda)
    C.orca_linear(C.ORCA_DTYPE_BF16, C.ORCA_LINEAR_F32OUT, A.data_ptr(), W.data_ptr(), 0, out.data_ptr(), M, N, K,
                  status.data_ptr(), torch.cuda.current_stream().cuda_stream, scratch_ptr=scratch.data_ptr(),
                  scratch_bytes=64 << 20, argmax_ptr=keys.data_ptr())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = [C.argmax_key_column(k) for k in keys.cpu().numpy().tolist()]
    want = np.argmax(out.cpu().numpy(), axis=1).tolist()
    assert got == want


# ------------------------------------------------------------------ toy fp32: Figure 5

def _toy_weights(seed=0):
    return synth.make_weights(synth.TOY, seed=seed, w_std=0.08, bias_std=0.02, ln_std=0.1)


def test_toy_fp32_figure5_greedy(cuda):
    """Toy GPT (2 layers, H=64, 4 heads, vocab 256), the four Figure 5
    requests; iteration 1 is the 7-row Figure 5 batch; greedy to iteration 8."""
    shape = synth.TOY
    w = _toy_weights()
    trace = synth.figure5_trace(vocab=shape.vocab, seed=0, out_len=8, extra=10)
    from iteration_level_selective_gb300 import runtime as rt
    from iteration_level_selective_gb300 import _orca as C
    dev = cuda
    dw = rt.DeviceWeights(shape, dev, host=w)
    eng = rt.Engine(shape, dw, max_bs=4, n_slots=64, max_rows=64, device=dev)
    pool = rt.RequestPool(trace)
    loop = rt.ServingLoop(eng, pool, keep_logits=True)
    recs = [loop.step()]
    recs.append(loop.step())
    desc = C.orca_last_descriptor(eng.handle, 64)
    # Figure 5: x1 decode (3 cached), x2 decode (1 cached), x3 prefill 2, x4 prefill 3 -> 7 rows
    lay = oragged.layout([(1, 3), (1, 1), (2, 0), (3, 0)])
    assert recs[1].req_ids == [0, 1, 2, 3]
    assert recs[1].n_new == [1, 1, 2, 3] and recs[1].n_ctx == [3, 1, 0, 0]
    assert desc["n_rows"] == 7 and desc["row_off"] == lay["row_off"] == [0, 1, 2, 4, 7]
    assert desc["row_pos"] == lay["row_pos"] and desc["last_row"] == lay["last_row"]
    bases = recs[1].slot_base
    assert desc["row_slot"] == [bases[lay["row_req"][r]] + lay["row_pos"][r] for r in range(7)]
    recs += loop.run()
    assert recs[-1].it == 8
    hz.compare_schedule(recs, trace, max_bs=4, n_slots=64)
    got_tok = hz.gpu_tokens_by_request(recs)
    got_lg = hz.gpu_logits_by_request(recs)
    for req in trace:
        greedy, logits = hz.oracle_generate(shape, w, req, teacher_force=False)
        assert got_tok[req.req_id] == greedy, (req.req_id, got_tok[req.req_id], greedy)
        assert pool.tokens[[r.req_id for r in pool.reqs].index(req.req_id)][req.n_prompt:].tolist() == greedy
        for k, (g, o) in enumerate(zip(got_lg[req.req_id], logits)):
            assert hz.max_rel_err(g, o) < FP32_TOL, (req.req_id, k, hz.max_rel_err(g, o))


def test_toy_fp32_teacher_forced_poisson_trace(cuda):
    """12 requests, Poisson arrivals, max_bs 4 so requests wait and join
    mid-flight; slots tight enough that reservations break."""
    shape = synth.TOY
    w = _toy_weights(seed=3)
    trace = synth.make_trace(12, (1, 20), (1, 12), vocab=shape.vocab, seed=5, rate_per_iter=0.7, forced=True)
    n_slots = 60
    recs, eng, pool = hz.run_gpu(shape, w, trace, max_bs=4, n_slots=n_slots, max_rows=64, teacher_force=True,
                                 keep_all=True)
    hz.compare_schedule(recs, trace, max_bs=4, n_slots=n_slots)
    got_lg = hz.gpu_logits_by_request(recs)
    got_tok = hz.gpu_tokens_by_request(recs)
    for req in trace:
        greedy, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
        assert len(got_lg[req.req_id]) == len(logits) == hz.n_generated(req)
        for g, o in zip(got_lg[req.req_id], logits):
            assert hz.max_rel_err(g, o) < FP32_TOL
        assert got_tok[req.req_id] == greedy


@pytest.mark.parametrize("policy", [1, 2])
def test_toy_fp32_reservation_policies_tight_memory(cuda, policy):
    """Pow2 and Oracle reservations (CS349D Lecture 2, section 6.1) on a
    trace whose slots bind: the schedule, the slot bases and the K/V usage
    match the oracle scheduler; every request writes only inside the slots
    it reserved, and its logits equal its own generation."""
    from iteration_level_selective_gb300 import _orca as C
    shape = synth.TOY
    w = _toy_weights(seed=9)
    trace = synth.make_trace(12, (1, 20), (1, 12), vocab=shape.vocab, seed=10, rate_per_iter=1.0, forced=True,
                             max_extra=30)
    n_slots = 64
    recs, eng, pool = hz.run_gpu(shape, w, trace, max_bs=6, n_slots=n_slots, max_rows=64, teacher_force=True,
                                 keep_all=True, reserve_policy=policy)
    hz.compare_schedule(recs, trace, max_bs=6, n_slots=n_slots, reserve_policy=policy)
    mx = osched.run_schedule(trace, max_bs=6, n_slots=n_slots, policy=osched.RESERVE_MAX)
    assert len(recs) < len(mx)  # smaller reservations admit more requests at once
    assert C.orca_kv_usage(eng.handle, pool.arr, pool.n) == (0, 0)  # all finished, all released
    got_lg = hz.gpu_logits_by_request(recs)
    for req in trace:
        _, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
        assert len(got_lg[req.req_id]) == len(logits)
        for g, o in zip(got_lg[req.req_id], logits):
            assert hz.max_rel_err(g, o) < FP32_TOL


# ------------------------------------------------------------------ bf16, multi-tile

SMALL_BF16 = synth.ModelShape(n_layers=2, hidden=256, n_heads=4, ffn=1024, vocab=1000, max_pos=1024,
                              dtype=synth.DTYPE_BF16)


def test_small_bf16_mixed_prefill_decode_multi_tile(cuda):
    """bf16 model with several GEMM tiles and ragged tails (rows ~ 1.3k,
    N = 768/256/1024/1000), prefills of up to 600 tokens (38 query tiles)
    and decode rows with > 256 keys (several key splits merged)."""
    shape = SMALL_BF16
    w = synth.make_weights(shape, seed=11, w_std=0.05, bias_std=0.02, ln_std=0.1)
    trace = synth.make_trace(6, (1, 600), (2, 9), vocab=shape.vocab, seed=12, rate_per_iter=0.5, forced=True)
    recs, eng, pool = hz.run_gpu(shape, w, trace, max_bs=8, n_slots=8000, max_rows=2048, teacher_force=True,
                                 keep_all=True)
    hz.compare_schedule(recs, trace, max_bs=8, n_slots=8000)
    got_lg = hz.gpu_logits_by_request(recs)
    worst = 0.0
    for req in trace:
        _, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
        for g, o in zip(got_lg[req.req_id], logits):
            worst = max(worst, hz.max_rel_err(g, o))
    assert worst < BF16_TOL, worst


# ------------------------------------------------------------------ chunked prefill under a token budget

@pytest.mark.parametrize("which", ["toy_fp32", "small_bf16"])
def test_chunked_prefill_token_budget(cuda, which):
    """Prompts cut into chunks under a per-iteration token budget (decode
    first): the integer record is bit-exact against the oracle scheduler,
    and each request's logits equal its own token-at-a-time generation
    (chunking changes no result), under teacher forcing.  The bf16 case has
    64-row chunks with cached context (tensor-core prompt attention) and
    shorter tails (CUDA-core query tiles)."""
    if which == "toy_fp32":
        shape, w, tol = synth.TOY, _toy_weights(seed=7), FP32_TOL
        trace = synth.make_trace(10, (1, 40), (1, 8), vocab=shape.vocab, seed=8, rate_per_iter=0.8, forced=True)
        kw = dict(max_bs=4, n_slots=200, max_rows=64, token_budget=12, chunk=5)
    else:
        shape, tol = SMALL_BF16, BF16_TOL
        w = synth.make_weights(shape, seed=31, w_std=0.05, bias_std=0.02, ln_std=0.1)
        trace = synth.make_trace(10, (1, 400), (1, 8), vocab=shape.vocab, seed=32, rate_per_iter=0.7, forced=True)
        kw = dict(max_bs=8, n_slots=8000, max_rows=2048, token_budget=150, chunk=64)
    recs, eng, pool = hz.run_gpu(shape, w, trace, teacher_force=True, keep_all=True, **kw)
    hz.compare_schedule(recs, trace, max_bs=kw["max_bs"], n_slots=kw["n_slots"], token_budget=kw["token_budget"],
                        chunk=kw["chunk"])
    assert max(sum(r.n_new) for r in recs) <= kw["token_budget"]
    assert any(c > 0 and L > 1 for r in recs for L, c in zip(r.n_new, r.n_ctx))  # chunks with cached context
    got_lg = hz.gpu_logits_by_request(recs)
    got_tok = hz.gpu_tokens_by_request(recs)
    worst = 0.0
    for req in trace:
        greedy, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
        assert len(got_lg[req.req_id]) == len(logits) == hz.n_generated(req)
        for g, o in zip(got_lg[req.req_id], logits):
            worst = max(worst, hz.max_rel_err(g, o))
        if which == "toy_fp32":
            assert got_tok[req.req_id] == greedy
    assert worst < tol, worst


# ------------------------------------------------------------------ paged K/V

@pytest.mark.parametrize("which", ["toy_fp32", "small_bf16"])
def test_paged_kv_with_preemption(cuda, which):
    """Paged K/V (blocks of 32 slots handed out as requests grow) in a pool
    small enough that requests are preempted and recomputed: the integer
    record (batches, rows, preemptions, releases) matches the oracle, and
    every request's logits equal its own generation - the recomputation
    after a preemption changes no result.  The bf16 case runs prompts on the
    tensor-core attention (K/V tiles gathered block by block) and decode
    rows with key splits over block runs."""
    from iteration_level_selective_gb300 import _orca as C
    if which == "toy_fp32":
        shape, w, tol = synth.TOY, _toy_weights(seed=17), FP32_TOL
        trace = synth.make_trace(10, (1, 40), (1, 20), vocab=shape.vocab, seed=18, rate_per_iter=1.5, forced=True)
        kw = dict(max_bs=4, n_slots=4 * 32, max_rows=256)
    else:
        shape, tol = SMALL_BF16, BF16_TOL
        w = synth.make_weights(shape, seed=19, w_std=0.05, bias_std=0.02, ln_std=0.1)
        trace = synth.make_trace(10, (1, 160), (10, 60), vocab=shape.vocab, seed=20, rate_per_iter=1.5, forced=True)
        kw = dict(max_bs=6, n_slots=6 * 32, max_rows=2048)
    pol = C.ORCA_RESERVE_PAGED
    recs, eng, pool = hz.run_gpu(shape, w, trace, teacher_force=True, keep_all=True, reserve_policy=pol, **kw)
    hz.compare_schedule(recs, trace, max_bs=kw["max_bs"], n_slots=kw["n_slots"], reserve_policy=pol)
    assert any(r.preempted for r in recs)
    got_lg = hz.gpu_logits_by_request(recs)
    worst = 0.0
    for req in trace:
        _, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
        assert len(got_lg[req.req_id]) == len(logits)
        for g, o in zip(got_lg[req.req_id], logits):
            worst = max(worst, hz.max_rel_err(g, o))
    assert worst < tol, worst
    assert C.orca_kv_usage(eng.handle, pool.arr, pool.n) == (0, 0)


# ------------------------------------------------------------------ two batches in flight

@pytest.mark.parametrize("which", ["toy_fp32", "small_bf16"])
def test_two_batches_in_flight(cuda, which):
    """Algorithm 1 with n_workers = 2: the next batch is selected from the
    requests not RUNNING and enqueued while the previous one runs.  The
    integer record matches the oracle's two-worker schedule and every
    request's logits equal its own generation (teacher forcing)."""
    if which == "toy_fp32":
        shape, w, tol = synth.TOY, _toy_weights(seed=13), FP32_TOL
        trace = synth.make_trace(12, (1, 20), (1, 12), vocab=shape.vocab, seed=14, rate_per_iter=0.8, forced=True)
        kw = dict(max_bs=4, n_slots=300, max_rows=64)
    else:
        shape, tol = SMALL_BF16, BF16_TOL
        w = synth.make_weights(shape, seed=15, w_std=0.05, bias_std=0.02, ln_std=0.1)
        trace = synth.make_trace(12, (1, 300), (1, 10), vocab=shape.vocab, seed=16, rate_per_iter=0.8, forced=True)
        kw = dict(max_bs=6, n_slots=8000, max_rows=2048)
    recs, eng, pool = hz.run_gpu(shape, w, trace, teacher_force=True, keep_all=True, n_workers=2, **kw)
    hz.compare_schedule(recs, trace, max_bs=kw["max_bs"], n_slots=kw["n_slots"], n_workers=2)
    got_lg = hz.gpu_logits_by_request(recs)
    worst = 0.0
    for req in trace:
        _, logits = hz.oracle_generate(shape, w, req, teacher_force=True)
        assert len(got_lg[req.req_id]) == len(logits)
        for g, o in zip(got_lg[req.req_id], logits):
            worst = max(worst, hz.max_rel_err(g, o))
    assert worst < tol, worst


def test_in_flight_limits(cuda):
    """At most two iterations in flight, never sharing a request."""
    import ctypes
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import runtime as rt
    shape = synth.TOY
    dw = rt.DeviceWeights(shape, cuda, host=_toy_weights())
    eng = rt.Engine(shape, dw, max_bs=4, n_slots=200, max_rows=64, device=cuda)
    trace = synth.make_trace(3, (2, 4), (3, 3), vocab=shape.vocab, seed=1)
    pool = rt.RequestPool(trace)
    st = torch.cuda.current_stream().cuda_stream
    bi = (ctypes.c_int32 * 4)()
    nt = (ctypes.c_int32 * 4)()
    one = (ctypes.c_int32 * 1)
    nb = C.orca_select_batch(eng.handle, pool.arr, 1, bi)   # request 0
    C.orca_iteration_submit(eng.handle, pool.arr, one(0), 1, 0, 0, st)
    with pytest.raises(C.OrcaError) as ei:                  # request 0 again while in flight
        C.orca_iteration_submit(eng.handle, pool.arr, one(0), 1, 0, 0, st)
    assert ei.value.code == C.ORCA_EINVAL
    assert C.orca_select_batch(eng.handle, pool.arr, 3, bi) == 2   # requests 1 and 2
    C.orca_iteration_submit(eng.handle, pool.arr, one(1), 1, 0, 0, st)
    with pytest.raises(C.OrcaError) as ei:                  # a third in flight
        C.orca_iteration_submit(eng.handle, pool.arr, one(2), 1, 0, 0, st)
    assert ei.value.code == C.ORCA_ESTATE
    with pytest.raises(C.OrcaError) as ei:                  # synchronous call while two are in flight
        C.orca_iteration(eng.handle, pool.arr, one(2), 1, 0, nt)
    assert ei.value.code == C.ORCA_ESTATE
    assert C.orca_iteration_wait(eng.handle, bi, nt) == 1 and bi[0] == 0
    assert C.orca_iteration_wait(eng.handle, bi, nt) == 1 and bi[0] == 1
    assert pool.view["n_generated"].tolist() == [1, 1, 0] and nb == 1
    eng.close()


def test_graph_replay_equals_eager_launches(cuda):
    """The CUDA-graph replay (sizes read from the device descriptor, fixed
    grids) and eager launches run the same decompositions: identical logits
    and tokens, iteration by iteration, over a trace whose batches change
    shape every iteration."""
    shape = SMALL_BF16
    w = synth.make_weights(shape, seed=21, w_std=0.05, bias_std=0.02, ln_std=0.1)
    trace = synth.make_trace(10, (1, 300), (1, 12), vocab=shape.vocab, seed=22, rate_per_iter=0.6, forced=True)
    out = []
    for eager in (False, True):
        recs, eng, pool = hz.run_gpu(shape, w, trace, max_bs=8, n_slots=8000, max_rows=2048, teacher_force=True,
                                     keep_all=True, eager=eager)
        out.append(recs)
        eng.close()
    assert len(out[0]) == len(out[1])
    nl = shape.n_layers
    for g, e in zip(*out):
        assert g.req_ids == e.req_ids and g.next_tokens == e.next_tokens
        np.testing.assert_array_equal(g.logits, e.logits)
        # embed (with the first LN1), final LN, LM head + per layer QKV (LN1
        # folded in), attention, Attn-Out, FC1 (LN2 folded in), FC2, and the
        # tensor-core prompt attention when a prompt of >= 32 rows is in the
        # batch
        want = 3 + nl * (5 + int(max(e.n_new) >= 32))
        assert g.launches == want and e.launches == want


def test_launch_stamps_time_the_graph_path(cuda):
    """Profiling mode 2 (launch stamps in the graph-replayed forward): the
    tokens and logits are those of an unprofiled run, every launch of every
    iteration is counted in its class, and the classes' times add up to no
    more than the device time of the iterations (CUDA events around them)."""
    from iteration_level_selective_gb300 import _orca as C
    from iteration_level_selective_gb300 import runtime as rt
    shape = SMALL_BF16
    w = synth.make_weights(shape, seed=21, w_std=0.05, bias_std=0.02, ln_std=0.1)
    trace = synth.make_trace(10, (1, 300), (1, 12), vocab=shape.vocab, seed=22, rate_per_iter=0.6, forced=True)
    out = []
    for mode in (0, 2, 1):
        dw = rt.DeviceWeights(shape, cuda, host=w)
        eng = rt.Engine(shape, dw, max_bs=8, n_slots=8000, max_rows=2048, device=cuda)
        C.orca_profile_enable(eng.handle, mode)
        loop = rt.ServingLoop(eng, rt.RequestPool(trace, teacher_force=True), teacher_force=True, keep_logits=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(loop.stream)
        recs = loop.run()
        e1.record(loop.stream)
        torch.cuda.synchronize()
        stats = {C.KERNEL_NAMES[k]: C.orca_profile_read(eng.handle, k) for k in range(C.ORCA_K_COUNT)}
        out.append((recs, stats, e0.elapsed_time(e1)))
        eng.close()
    (r0, _, _), (r2, stats, dev_ms), (r1, stats1, dev_ms1) = out
    # mode 2 keeps the graph path (the eager event mode is launch-bound on this small model)
    assert dev_ms < 0.9 * dev_ms1, (dev_ms, dev_ms1)
    for a, b in zip(r0, r2):
        assert a.next_tokens == b.next_tokens
        np.testing.assert_array_equal(a.logits, b.logits)
    n_it, nl = len(r2), shape.n_layers
    # embed, final LN, LM head; per layer QKV, attention (both launches: one stamp), Attn-Out, FC1, FC2
    assert stats["embed"]["launches"] == n_it and stats["lm_head"]["launches"] == n_it
    assert stats["layernorm"]["launches"] == n_it
    for k in ("gemm_qkv", "attention", "gemm_o", "gemm_fc1", "gemm_fc2"):
        assert stats[k]["launches"] == n_it * nl, k
        assert stats[k]["total_ms"] > 0 and stats[k]["flops"] > 0, k
    total = sum(s["total_ms"] for s in stats.values())
    assert 0 < total <= dev_ms, (total, dev_ms)


# ------------------------------------------------------------------ GPT-2-small, full size, sampled

def test_gpt2_small_trace_sampled_parity(cuda):
    """GPT-2-small-shaped bf16 model (12 layers, H=768, 12 heads, vocab
    50257), 64 requests, prompts U{32..512}, outputs U{1..256},
    max_tokens = prompt + 256, max_bs 64 - the benchmark's workload and
    launch configuration.  Teacher-forced; the integer schedule is checked
    in full and, against the oracle, the logits of the three shortest-prompt
    requests at up to 6 generated steps and of two requests with prompts of
    256-400 rows (prompt attention on the tensor cores) at up to 2."""
    shape = synth.GPT2_SMALL
    w = synth.make_weights(shape, seed=0)
    trace = synth.make_trace(64, (32, 512), (1, 256), vocab=shape.vocab, seed=0, rate_per_iter=0.5,
                             max_extra=256, forced=True)
    by_len = sorted(trace, key=lambda r: r.n_prompt)
    # the three shortest prompts, and two of 256-400 rows: their prompt iteration runs the
    # tensor-core prompt attention (>= 32 rows) next to the batch's decode rows
    long = [r for r in by_len if 256 <= r.n_prompt <= 400][:2]
    assert len(long) == 2
    sample = by_len[:3] + long
    n_slots = 64 * (512 + 256)
    recs, eng, pool = hz.run_gpu(shape, w, trace, max_bs=64, n_slots=n_slots, max_rows=64 * 512,
                                 teacher_force=True, keep_ids={r.req_id for r in sample})
    hz.compare_schedule(recs, trace, max_bs=64, n_slots=n_slots)
    got_lg = hz.gpu_logits_by_request(recs)
    for req in sample:
        steps = min(6 if req.n_prompt < 256 else 2, hz.n_generated(req))
        _, logits = hz.oracle_generate(shape, w, req, teacher_force=True, stop_after=steps)
        for k in range(steps):
            err = hz.max_rel_err(got_lg[req.req_id][k], logits[k])
            assert err < BF16_TOL, (req.req_id, k, err)


# ------------------------------------------------------------------ edge cases

def test_iteration_errors_leave_requests_untouched(cuda):
    from iteration_level_selective_gb300 import runtime as rt
    from iteration_level_selective_gb300 import _orca as C
    import ctypes
    shape = synth.TOY
    dw = rt.DeviceWeights(shape, cuda, host=_toy_weights())
    eng = rt.Engine(shape, dw, max_bs=2, n_slots=64, max_rows=8, device=cuda)
    trace = synth.make_trace(3, (5, 5), (2, 2), vocab=256, seed=1)
    pool = rt.RequestPool(trace)
    bi = (ctypes.c_int32 * 2)()
    nt = (ctypes.c_int32 * 2)()
    nb = C.orca_select_batch(eng.handle, pool.arr, 3, bi)
    assert nb == 2
    with pytest.raises(C.OrcaError) as ei:    # 5 + 5 rows > max_rows 8
        C.orca_iteration(eng.handle, pool.arr, bi, nb, 0, nt)
    assert ei.value.code == C.ORCA_EBATCH
    assert pool.arr[bi[0]].state == C.ORCA_RUNNING and pool.arr[bi[0]].n_cached == 0
    with pytest.raises(C.OrcaError) as ei:
        C.orca_iteration(eng.handle, pool.arr, bi, 0, 0, nt)
    assert ei.value.code == C.ORCA_EINVAL
    pool.tokens[0][0] = 999                   # token id out of range
    with pytest.raises(C.OrcaError) as ei:
        C.orca_iteration(eng.handle, pool.arr, bi, 1, 0, nt)
    assert ei.value.code == C.ORCA_EINVAL
    pool.tokens[0][0] = 1
    C.orca_iteration(eng.handle, pool.arr, bi, 1, 0, nt)   # one request fits
    assert pool.arr[bi[0]].n_cached == 5 and pool.arr[bi[0]].state == C.ORCA_INCREMENT

"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own code: printed worked
examples (tests/golden), library routines (torch layer_norm, gelu,
scaled_dot_product_attention, bf16 conversion), closed forms and brute force.
A few tests plant a mistake in the oracle to show that a pin catches it.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import model as omodel
from oracle import numerics, ragged, scheduler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows, expect = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] in ("n_rows", "padded_rows", "useful_pairs", "padded_pairs", "max_bs",
                            "iterations"):
                expect[parts[0]] = int(parts[1])
            else:
                rows.append(parts)
    return rows, expect


# ---------------------------------------------------------------- numerics

def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        # exact ties between two bf16 values: 1 + k/256 + 1/512
                        1.0 + np.arange(0, 64) / 256.0 + 1.0 / 512.0,
                        -(2.0 + np.arange(0, 64) / 128.0 + 1.0 / 256.0)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = numerics.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_layer_norm_matches_torch():
    rng = np.random.default_rng(2)
    x, g, b = rng.standard_normal((7, 96)), rng.standard_normal(96), rng.standard_normal(96)
    want = F.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), torch.from_numpy(b),
                        eps=1e-5).numpy()
    np.testing.assert_allclose(numerics.layer_norm(x, g, b), want, rtol=1e-12, atol=1e-12)


def test_gelu_matches_torch_tanh_form():
    x = np.linspace(-8, 8, 4001)
    want = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(numerics.gelu_tanh(x), want, rtol=1e-13, atol=1e-15)


def test_softmax_sums_to_one_and_is_shift_invariant():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((5, 33)) * 30
    p = numerics.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(numerics.softmax(s + 123.0), p, rtol=1e-12)
    # brute force against the definition exp(s)/sum exp(s) in a safe range
    s2 = rng.standard_normal(9)
    np.testing.assert_allclose(numerics.softmax(s2), np.exp(s2) / np.exp(s2).sum(), rtol=1e-14)


# ---------------------------------------------------------------- forward math

def _torch_full_forward(shape, w, tokens, bf16):
    """Whole-sequence causal GPT forward from torch library routines: the
    same model computed all positions at once instead of token by token."""
    R = (lambda t: t.to(torch.bfloat16).to(torch.float64)) if bf16 else (lambda t: t)
    T_ = lambda k: torch.from_numpy(np.asarray(w[k], dtype=np.float64))
    H, nh = shape.hidden, shape.n_heads
    d = H // nh
    T = len(tokens)
    ids = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
    x = T_("tok_emb")[ids] + T_("pos_emb")[:T]
    for l in range(shape.n_layers):
        p = lambda k: T_(f"L{l}.{k}")
        h = R(F.layer_norm(x, (H,), p("ln1_g"), p("ln1_b"), eps=1e-5))
        q, k, v = R(F.linear(h, p("w_qkv"), p("b_qkv"))).split(H, dim=-1)
        heads = lambda t: t.view(T, nh, d).transpose(0, 1)
        a = F.scaled_dot_product_attention(heads(q), heads(k), heads(v), is_causal=True)
        a = R(a.transpose(0, 1).reshape(T, H))
        x = x + F.linear(a, p("w_o"), p("b_o"))
        h2 = R(F.layer_norm(x, (H,), p("ln2_g"), p("ln2_b"), eps=1e-5))
        u = R(F.gelu(F.linear(h2, p("w_fc1"), p("b_fc1")), approximate="tanh"))
        x = x + F.linear(u, p("w_fc2"), p("b_fc2"))
    hf = R(F.layer_norm(x, (H,), T_("lnf_g"), T_("lnf_b"), eps=1e-5))
    return (hf @ T_("tok_emb").T).numpy()


def _gen_vs_full(shape, seed, n_prompt, out_len, w_std=0.08):
    w = synth.make_weights(shape, seed=seed, w_std=w_std, bias_std=0.05, ln_std=0.2)
    rng = np.random.default_rng(seed)
    prompt = rng.integers(0, shape.vocab, n_prompt)
    forced = rng.integers(0, shape.vocab, out_len)
    orc = omodel.GPTOracle(shape, w)
    greedy, logits, fed = orc.generate(prompt, out_len, forced=forced)
    seq = np.concatenate([prompt, forced[:out_len - 1]])
    full = _torch_full_forward(shape, w, seq, shape.dtype == synth.DTYPE_BF16)
    want = full[n_prompt - 1:]
    return np.stack(logits), want, greedy


def test_generation_equals_full_sequence_forward_fp32():
    got, want, greedy = _gen_vs_full(synth.TOY, seed=5, n_prompt=6, out_len=9)
    assert got.shape == want.shape == (9, synth.TOY.vocab)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-11 * np.abs(want).max())
    assert greedy == list(np.argmax(want, axis=-1))


def test_generation_equals_full_sequence_forward_bf16_rounding_points():
    shape = synth.with_dtype(synth.TOY, synth.DTYPE_BF16)
    got, want, _ = _gen_vs_full(shape, seed=6, n_prompt=5, out_len=6)
    # the two sides round the same fp64 values to bf16 (torch goes through
    # fp32 first); a rare double-rounding tie may move one bf16 ulp.
    err = np.abs(got - want).max() / np.abs(want).max()
    assert err < 1e-3, err


def test_single_token_attention_returns_value_exactly():
    # one key: softmax = 1, so attention returns V (closed form)
    orc = omodel.GPTOracle(synth.TOY, synth.make_weights(synth.TOY, seed=1))
    rng = np.random.default_rng(4)
    q, K, V = rng.standard_normal(64), rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    np.testing.assert_array_equal(orc.attend(q, K, V), V[0])


def test_attend_matches_sdpa_for_one_query():
    orc = omodel.GPTOracle(synth.TOY, synth.make_weights(synth.TOY, seed=1))
    rng = np.random.default_rng(7)
    T = 37
    q, K, V = rng.standard_normal(64) * 3, rng.standard_normal((T, 64)) * 3, rng.standard_normal((T, 64))
    hq = torch.from_numpy(q).view(1, 4, 16).transpose(0, 1)       # [h, 1, d]
    hk = torch.from_numpy(K).view(T, 4, 16).transpose(0, 1)       # [h, T, d]
    hv = torch.from_numpy(V).view(T, 4, 16).transpose(0, 1)
    want = F.scaled_dot_product_attention(hq, hk, hv).transpose(0, 1).reshape(64).numpy()
    np.testing.assert_allclose(orc.attend(q, K, V), want, rtol=1e-12, atol=1e-13)


def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible mistakes in the oracle; the full-forward pin must fail."""
    base_attend = omodel.GPTOracle.attend

    def wrong_scale(self, q, K, V):
        return base_attend(self, q * np.sqrt(self.d), K, V)   # softmax scale dropped

    def off_by_one(self, q, K, V):
        return base_attend(self, q, K[:-1], V[:-1]) if len(K) > 1 else base_attend(self, q, K, V)

    for bad in (wrong_scale, off_by_one):
        monkeypatch.setattr(omodel.GPTOracle, "attend", bad)
        got, want, _ = _gen_vs_full(synth.TOY, seed=5, n_prompt=6, out_len=4)
        assert np.abs(got - want).max() > 1e-6 * np.abs(want).max()
        monkeypatch.setattr(omodel.GPTOracle, "attend", base_attend)
    # a dropped bias in the MLP
    base_gelu = omodel.gelu_tanh
    monkeypatch.setattr(omodel, "gelu_tanh", lambda z: base_gelu(z) * 1.01)
    got, want, _ = _gen_vs_full(synth.TOY, seed=5, n_prompt=6, out_len=4)
    assert np.abs(got - want).max() > 1e-6 * np.abs(want).max()


def test_causality_future_tokens_do_not_change_past_logits():
    w = synth.make_weights(synth.TOY, seed=9, w_std=0.08)
    orc = omodel.GPTOracle(synth.TOY, w)
    rng = np.random.default_rng(9)
    prompt = rng.integers(0, 256, 5)
    f1 = rng.integers(0, 256, 6)
    f2 = f1.copy()
    f2[3:] = (f2[3:] + 17) % 256
    _, l1, _ = orc.generate(prompt, 6, forced=f1)
    _, l2, _ = orc.generate(prompt, 6, forced=f2)
    for k in range(4):      # logits k depend on forced[:k] only
        np.testing.assert_array_equal(l1[k], l2[k])
    assert not np.array_equal(l1[5], l2[5])


# ---------------------------------------------------------------- ragged layout

def test_figure5_layout():
    rows, expect = _read_golden("figure5_batch.txt")
    batch = [(int(L), int(c)) for _, L, c in rows]
    lay = ragged.layout(batch)
    assert lay["n_rows"] == expect["n_rows"] == 7
    assert lay["row_off"] == [0, 1, 2, 4, 7]
    assert lay["row_pos"] == [3, 1, 0, 1, 0, 1, 2]
    assert lay["last_row"] == [0, 1, 3, 6]
    assert ragged.padded_rows(batch) == expect["padded_rows"]
    # brute force over an explicit causal mask: 4 + 2 + 3 + 6 pairs per head
    pairs = sum(1 for r in range(7) for key in range(lay["row_pos"][r] + 1))
    assert ragged.useful_pairs(batch) == pairs == 15


def test_exercise4_counts():
    rows, expect = _read_golden("exercise4_counts.txt")
    batch = [(int(L), int(c)) for L, c in rows]
    assert ragged.layout(batch)["n_rows"] == expect["n_rows"]
    assert ragged.padded_rows(batch) == expect["padded_rows"]
    assert ragged.useful_pairs(batch) == expect["useful_pairs"]
    assert ragged.padded_pairs(batch) == expect["padded_pairs"]
    assert round(expect["padded_pairs"] / expect["useful_pairs"], 1) == 23.6


# ---------------------------------------------------------------- scheduler

class _R:
    def __init__(self, req_id, arrival, n_prompt, out_len, max_tokens):
        self.req_id, self.arrival, self.n_prompt = req_id, arrival, n_prompt
        self.out_len, self.max_tokens = out_len, max_tokens


def _timeline_from_records(records, n_req):
    last_it = max(r.it for r in records)
    grid = {i: [" "] * (last_it + 1) for i in range(n_req)}
    for rec in records:
        for rid, L, c in zip(rec.req_ids, rec.n_new, rec.n_ctx):
            grid[rid][rec.it] = "P" if c == 0 else "D"
    return grid


def test_demo4_timeline():
    rows, expect = _read_golden("demo4_timeline.txt")
    # generated tokens = number of P/D cells; prompt length is irrelevant to the schedule
    trace = []
    for name, arrival, line in rows:
        n_out = sum(ch in "PD" for ch in line)
        trace.append(_R(int(name[1:]), int(arrival), 4, n_out, 4 + n_out))
    recs = scheduler.run_schedule(trace, max_bs=expect["max_bs"], n_slots=10_000)
    assert len(recs) == expect["iterations"] == 10
    grid = _timeline_from_records(recs, len(trace))
    for name, arrival, line in rows:
        i = int(name[1:])
        want = line.replace("_", " ").replace(".", " ")
        got = "".join(grid[i]).rstrip()
        assert got == want.rstrip(), (name, got, want)
        # waiting cells: arrived, not scheduled
        for t, ch in enumerate(line):
            if ch == ".":
                assert t >= int(arrival) and grid[i][t] == " "


def test_break_stops_selection_no_skipping():
    # head request does not fit: later, smaller requests must not be admitted
    slots = scheduler.SlotPool(10)
    pool = [scheduler.ReqState(0, 0, 2, 5, 8), scheduler.ReqState(1, 1, 2, 2, 4),
            scheduler.ReqState(2, 2, 1, 1, 2)]
    b = scheduler.select(pool, slots, max_bs=8)
    assert [r.req_id for r in b] == [0] and slots.n_rsrv == 8
    # request 0 keeps running; 1 still does not fit (8 + 4 > 10) so 2 waits too
    pool[0].state = scheduler.INCREMENT
    b = scheduler.select(pool, slots, max_bs=8)
    assert [r.req_id for r in b] == [0] and slots.n_rsrv == 8
    slots.release(0)
    pool[0].state = scheduler.FINISHED
    b = scheduler.select(pool, slots, max_bs=8)
    assert [r.req_id for r in b] == [1, 2] and slots.n_rsrv == 6
    assert [r.slot_base for r in b] == [0, 4]


def test_max_bs_stops_before_reserving():
    slots = scheduler.SlotPool(100)
    pool = [scheduler.ReqState(i, 0, 2, 2, 5) for i in range(5)]
    b = scheduler.select(pool, slots, max_bs=3)
    assert [r.req_id for r in b] == [0, 1, 2] and slots.n_rsrv == 15
    assert [r.slot_base for r in pool] == [0, 5, 10, -1, -1]


def test_arrival_ties_break_by_request_id():
    slots = scheduler.SlotPool(100)
    pool = [scheduler.ReqState(7, 3, 2, 2, 5), scheduler.ReqState(2, 3, 2, 2, 5),
            scheduler.ReqState(5, 1, 2, 2, 5)]
    assert [r.req_id for r in scheduler.select(pool, slots, 8)] == [5, 2, 7]


def test_release_restores_reservation_and_merges_holes():
    s = scheduler.SlotPool(20)
    assert [s.reserve(i, n) for i, n in enumerate([5, 5, 5])] == [0, 5, 10]
    s.release(1)
    assert s.reserve(3, 6) is None and s.frag_blocks == 1      # count ok (16 <= 20), no hole of 6
    assert s.reserve(4, 5) == 5                                  # first fit, lowest base
    s.release(0), s.release(4), s.release(2)
    assert s.n_rsrv == 0 and s.free == [(0, 20)]
    with pytest.raises(KeyError):
        s.release(2)


def test_max_bs_one_is_sequential_serving():
    rng = np.random.default_rng(11)
    trace = [_R(i, int(a), int(rng.integers(1, 9)), int(rng.integers(1, 6)), 20)
             for i, a in enumerate(sorted(rng.integers(0, 30, 12)))]
    recs = scheduler.run_schedule(trace, max_bs=1, n_slots=1000)
    order = [r.req_ids[0] for r in recs]
    # each request runs all its iterations back to back, in arrival order
    expect = [t.req_id for t in sorted(trace, key=lambda t: (t.arrival, t.req_id)) for _ in range(t.out_len)]
    assert order == expect


def test_fcfs_invariant_and_reservation_bound_random_traces():
    rng = np.random.default_rng(12)
    for trial in range(30):
        n = int(rng.integers(5, 40))
        n_slots = int(rng.integers(30, 200))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 12)), int(rng.integers(1, 15))
            trace.append(_R(i, int(rng.integers(0, 40)), lp, lo, lp + lo + int(rng.integers(0, 5))))
        recs = scheduler.run_schedule(trace, max_bs=int(rng.integers(1, 9)), n_slots=n_slots)
        iters = {t.req_id: 0 for t in trace}
        arrival = {t.req_id: (t.arrival, t.req_id) for t in trace}
        mt = {t.req_id: t.max_tokens for t in trace}
        live, done = set(), set()
        for rec in recs:
            for rid in rec.req_ids:
                iters[rid] += 1
                live.add(rid)
            assert sum(mt[r] for r in live) <= n_slots
            # batch order is arrival order
            assert [arrival[r] for r in rec.req_ids] == sorted(arrival[r] for r in rec.req_ids)
            live -= set(rec.released)
            done |= set(rec.released)
            # iteration-level FCFS over the pool (arrived, unfinished requests)
            in_pool = [t.req_id for t in trace if t.arrival <= rec.it and t.req_id not in done]
            for a in in_pool:
                for b in in_pool:
                    if arrival[a] < arrival[b]:
                        assert iters[a] >= iters[b], (trial, rec.it, a, b)
        assert all(iters[t.req_id] == t.out_len for t in trace)


# ---------------------------------------------------------------- chunked prefill under a token budget
# CS349D Lecture 2, Exercise 9 (prompt chunks, SeqWork(n_new, n_past), a cap
# on the tokens of one iteration); static-to-continuous article, chunked
# prefill (decode first, the rest of the budget to prompt chunks).

def _records(recs):
    return [(r.it, r.req_ids, r.n_new, r.n_ctx, sorted(r.released)) for r in recs]


def test_budget_worked_example_by_hand():
    # A: prompt 5, B: prompt 3, both arrive at 0, 2 tokens each; budget 4,
    # chunk 3.
    #   it 0: no decodes; A takes min(5, 3, 4) = 3, B min(3, 3, 1) = 1
    #   it 1: no decodes; A takes min(2, 3, 4) = 2 (prompt done -> token 1),
    #         B min(2, 3, 2) = 2 (prompt done -> token 1)
    #   it 2: A and B decode one row each -> second token, both finish
    trace = [_R(0, 0, 5, 2, 7), _R(1, 0, 3, 2, 5)]
    recs = scheduler.run_schedule(trace, max_bs=4, n_slots=100, token_budget=4, chunk=3)
    assert _records(recs) == [(0, [0, 1], [3, 1], [0, 0], []),
                              (1, [0, 1], [2, 2], [3, 1], []),
                              (2, [0, 1], [1, 1], [5, 3], [0, 1])]


def test_budget_decodes_go_first():
    # A (prompt 2, 3 tokens) decodes from iteration 1; B (prompt 6) arrives
    # at 1.  Budget 3: each iteration A's decode row is served first and B
    # gets the 2 rows left (it 1: 2, it 2: 2); A finishes after it 2, so at
    # it 3 B takes its last 2 prompt rows alone.
    trace = [_R(0, 0, 2, 3, 5), _R(1, 1, 6, 1, 7)]
    recs = scheduler.run_schedule(trace, max_bs=4, n_slots=100, token_budget=3, chunk=8)
    assert _records(recs) == [(0, [0], [2], [0], []),
                              (1, [0, 1], [1, 2], [2, 0], []),
                              (2, [0, 1], [1, 2], [3, 2], [0]),
                              (3, [1], [2], [4], [1])]


def test_budget_admitted_request_keeps_reservation_while_idle():
    # budget 2 with two new prompts of 4: B is admitted (slots reserved by
    # Algorithm 1) but gets no row until A's prompt is done
    trace = [_R(0, 0, 4, 1, 5), _R(1, 0, 4, 1, 5)]
    order = sorted(trace, key=lambda r: (r.arrival, r.req_id))
    states = [scheduler.ReqState(r.req_id, r.arrival, r.n_prompt, r.out_len, r.max_tokens) for r in order]
    slots = scheduler.SlotPool(10)
    sel = scheduler.select_budget(states, slots, max_bs=4, token_budget=2, chunk=8)
    assert [(r.req_id, n) for r, n in sel] == [(0, 2), (1, 0)]
    assert slots.n_rsrv == 10 and states[1].slot_base == 5
    recs = scheduler.run_schedule(trace, max_bs=4, n_slots=10, token_budget=2, chunk=8)
    assert _records(recs) == [(0, [0], [2], [0], []), (1, [0], [2], [2], [0]),
                              (2, [1], [2], [0], []), (3, [1], [2], [2], [1])]


def test_unlimited_budget_is_algorithm_1():
    rng = np.random.default_rng(41)
    for trial in range(20):
        n = int(rng.integers(3, 30))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 12)), int(rng.integers(1, 10))
            trace.append(_R(i, int(rng.integers(0, 20)), lp, lo, lp + lo + int(rng.integers(0, 4))))
        kw = dict(max_bs=int(rng.integers(1, 9)), n_slots=int(rng.integers(30, 120)))
        plain = scheduler.run_schedule(trace, **kw)
        big = scheduler.run_schedule(trace, token_budget=2 ** 31 - 1, chunk=2 ** 31 - 1, **kw)
        assert _records(plain) == _records(big)
        assert [r.slot_base for r in plain] == [r.slot_base for r in big]


def test_budget_invariants_random_traces():
    rng = np.random.default_rng(42)
    for trial in range(30):
        n = int(rng.integers(3, 30))
        budget, chunk = int(rng.integers(1, 24)), int(rng.integers(1, 16))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 30)), int(rng.integers(1, 10))
            trace.append(_R(i, int(rng.integers(0, 20)), lp, lo, lp + lo + int(rng.integers(0, 4))))
        recs = scheduler.run_schedule(trace, max_bs=int(rng.integers(1, 9)), n_slots=400, token_budget=budget,
                                      chunk=chunk)
        n_prompt = {t.req_id: t.n_prompt for t in trace}
        done_prompt = {t.req_id: 0 for t in trace}
        generated = {t.req_id: 0 for t in trace}
        for rec in recs:
            assert 1 <= sum(rec.n_new) <= budget
            decoding = [c >= n_prompt[r] for r, c in zip(rec.req_ids, rec.n_ctx)]
            for rid, L, c, dec in zip(rec.req_ids, rec.n_new, rec.n_ctx, decoding):
                assert c == (done_prompt[rid] if not dec else n_prompt[rid] + generated[rid] - 1)
                if dec:
                    assert L == 1
                else:
                    assert 1 <= L <= min(chunk, n_prompt[rid] - c)
                    done_prompt[rid] += L
                if c + L >= n_prompt[rid]:
                    generated[rid] += 1
        assert done_prompt == n_prompt
        assert all(generated[t.req_id] == t.out_len for t in trace)


# ---------------------------------------------------------------- reservation variants (CS349D Lecture 2, 6.1)

def test_reserve_sizes_by_hand():
    R = scheduler.ReqState
    M, P2, O = scheduler.RESERVE_MAX, scheduler.RESERVE_POW2, scheduler.RESERVE_ORACLE
    size = scheduler.reserve_size
    r = R(0, 0, 300, 100, 556)          # true length 400
    assert (size(M, r), size(P2, r), size(O, r)) == (556, 512, 400)
    r = R(0, 0, 300, 300, 556)          # true length 600 > max_tokens: all capped
    assert (size(M, r), size(P2, r), size(O, r)) == (556, 556, 556)
    r = R(0, 0, 3, 2, 9)                # 5 -> 8
    assert (size(M, r), size(P2, r), size(O, r)) == (9, 8, 5)
    r = R(0, 0, 1, 1, 5)                # 2 is already a power of two
    assert (size(P2, r), size(O, r)) == (2, 2)


def test_tight_memory_policies_by_hand():
    # n_slots 10, A and B: prompt 2, 2 tokens, max_tokens 8 (true length 4).
    # Max: A takes 8 slots, B (8 more) does not fit and waits for A;
    # Pow2 and Oracle: 4 + 4 slots, both run together.
    trace = [_R(0, 0, 2, 2, 8), _R(1, 0, 2, 2, 8)]
    mx = scheduler.run_schedule(trace, max_bs=4, n_slots=10, policy=scheduler.RESERVE_MAX)
    assert _records(mx) == [(0, [0], [2], [0], []), (1, [0], [1], [2], [0]),
                            (2, [1], [2], [0], []), (3, [1], [1], [2], [1])]
    for pol in (scheduler.RESERVE_POW2, scheduler.RESERVE_ORACLE):
        recs = scheduler.run_schedule(trace, max_bs=4, n_slots=10, policy=pol)
        assert _records(recs) == [(0, [0, 1], [2, 2], [0, 0], []), (1, [0, 1], [1, 1], [2, 2], [0, 1])]
        assert recs[0].slot_base == [0, 4]


def test_policies_agree_when_memory_is_ample_and_stored_never_exceeds_reserved():
    rng = np.random.default_rng(43)
    for trial in range(20):
        n = int(rng.integers(3, 30))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 20)), int(rng.integers(1, 12))
            trace.append(_R(i, int(rng.integers(0, 20)), lp, lo, lp + lo + int(rng.integers(0, 20))))
        base = None
        for pol in (scheduler.RESERVE_MAX, scheduler.RESERVE_POW2, scheduler.RESERVE_ORACLE):
            recs = scheduler.run_schedule(trace, max_bs=int(trial % 7) + 1, n_slots=10_000, policy=pol)
            if base is None:
                base = _records(recs)
            assert _records(recs) == base
        # tight memory: at every step the written slots fit in the reservations
        for pol in (scheduler.RESERVE_MAX, scheduler.RESERVE_POW2, scheduler.RESERVE_ORACLE):
            order = sorted(trace, key=lambda r: (r.arrival, r.req_id))
            states = [scheduler.ReqState(r.req_id, r.arrival, r.n_prompt, r.out_len, r.max_tokens) for r in order]
            slots = scheduler.SlotPool(max(t.max_tokens for t in trace) * 2)
            for step in range(200):
                live = [r for r in states if r.arrival <= step and r.state != scheduler.FINISHED]
                if not live:
                    continue
                for r in scheduler.select(live, slots, 4, pol):
                    r.n_cached += scheduler.default_rows(r)
                    r.n_generated += 1
                    r.state = scheduler.INCREMENT
                    assert r.n_cached <= slots.owned[r.req_id][1]
                    if scheduler.finished(r):
                        r.state = scheduler.FINISHED
                        slots.release(r.req_id)
                reserved, stored = scheduler.kv_usage(states, slots)
                assert stored <= reserved <= slots.n_slots
            assert all(r.state == scheduler.FINISHED for r in states)


def test_kv_usage_reserved_vs_stored_by_hand():
    """CS349D Lecture 2, section 6.1: a reservation occupies slots that are
    not yet written ("reserved" is not "used").  Reading: after each
    iteration, reserved = slots held by reservations, stored = sum of the
    cached tokens of the requests that hold one.  Three requests, a 20-slot
    pool, max_bs 3:
        A: arrives 0, prompt 3, 4 tokens, max_tokens 10  (true length 7)
        B: arrives 0, prompt 2, 2 tokens, max_tokens 8   (true length 4)
        C: arrives 1, prompt 5, 3 tokens, max_tokens 12  (true length 8)
    Max reserves max_tokens: A 10 + B 8 = 18, so C (12) waits until A and B
    are both gone.
        it 0: A, B prefill            -> reserved 18, stored 3 + 2
        it 1: C does not fit (30 > 20); A 4 cached, B finishes (8 freed)
                                      -> 10, 4
        it 2: C still does not fit (22 > 20); A 5 cached      -> 10, 5
        it 3: A finishes              -> 0, 0
        it 4: C at base 0, prefill    -> 12, 5
        it 5, 6: C decodes, then finishes -> 12, 6 and 0, 0
    Pow2 reserves the true length rounded up to a power of two: A 8, B 4,
    C 8; Oracle the true length: A 7, B 4, C 8.  Both admit C at it 1.
        Pow2:   it 0 -> 12, 5; it 1 (B done, C prefills) -> 16, 4 + 5;
                it 2 -> 16, 5 + 6; it 3 (A and C done) -> 0, 0
        Oracle: it 0 -> 11, 5; it 1 -> 15, 9; it 2 -> 15, 11; it 3 -> 0, 0
    A mistake that sums n_prompt or max_tokens instead of the cached tokens,
    or that keeps a finished request's count, changes at least one pair."""
    trace = [_R(0, 0, 3, 4, 10), _R(1, 0, 2, 2, 8), _R(2, 1, 5, 3, 12)]
    want = {
        scheduler.RESERVE_MAX: [(0, [0, 1], (18, 5)), (1, [0, 1], (10, 4)), (2, [0], (10, 5)),
                                (3, [0], (0, 0)), (4, [2], (12, 5)), (5, [2], (12, 6)), (6, [2], (0, 0))],
        scheduler.RESERVE_POW2: [(0, [0, 1], (12, 5)), (1, [0, 1, 2], (16, 9)), (2, [0, 2], (16, 11)),
                                 (3, [0, 2], (0, 0))],
        scheduler.RESERVE_ORACLE: [(0, [0, 1], (11, 5)), (1, [0, 1, 2], (15, 9)), (2, [0, 2], (15, 11)),
                                   (3, [0, 2], (0, 0))],
    }
    for pol, rows in want.items():
        recs = scheduler.run_schedule(trace, max_bs=3, n_slots=20, policy=pol)
        assert [(r.it, r.req_ids, r.kv) for r in recs] == rows, pol
    # C lands at base 0 under Max (the two freed segments merged), at 12
    # under Pow2 (after A's 8 and B's 4) and at 11 under Oracle
    bases = {pol: {rid: b for r in scheduler.run_schedule(trace, max_bs=3, n_slots=20, policy=pol)
                   for rid, b in zip(r.req_ids, r.slot_base)}[2] for pol in want}
    assert bases == {scheduler.RESERVE_MAX: 0, scheduler.RESERVE_POW2: 12, scheduler.RESERVE_ORACLE: 11}


# ---------------------------------------------------------------- batches in flight (Algorithm 1, n_workers = 2)

def test_two_workers_by_hand():
    # A, B, C arrive at 0 (prompt 1, 2 tokens each), max_bs 2.  Iteration 0
    # schedules A, B; with one batch in flight the next Select sees only C;
    # then the oldest batch returns and A, B are selectable again, and so on.
    trace = [_R(0, 0, 1, 2, 3), _R(1, 0, 1, 2, 3), _R(2, 0, 1, 2, 3)]
    recs = scheduler.run_schedule(trace, max_bs=2, n_slots=100, n_workers=2)
    assert _records(recs) == [(0, [0, 1], [1, 1], [0, 0], []), (1, [2], [1], [0], []),
                              (2, [0, 1], [1, 1], [1, 1], [0, 1]), (3, [2], [1], [1], [2])]
    one = scheduler.run_schedule(trace, max_bs=2, n_slots=100, n_workers=1)
    assert _records(one) == [(0, [0, 1], [1, 1], [0, 0], []), (1, [0, 1], [1, 1], [1, 1], [0, 1]),
                             (2, [2], [1], [0], []), (3, [2], [1], [1], [2])]


def test_two_workers_invariants_random_traces():
    rng = np.random.default_rng(44)
    for trial in range(30):
        n = int(rng.integers(2, 30))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 12)), int(rng.integers(1, 10))
            trace.append(_R(i, int(rng.integers(0, 25)), lp, lo, lp + lo + int(rng.integers(0, 4))))
        kw = dict(max_bs=int(rng.integers(1, 9)), n_slots=int(rng.integers(30, 150)))
        if trial % 3 == 0:
            kw.update(token_budget=int(rng.integers(1, 20)), chunk=int(rng.integers(1, 10)))
        recs = scheduler.run_schedule(trace, n_workers=2, **kw)
        prompt_done = {t.req_id: 0 for t in trace}
        gen = {t.req_id: 0 for t in trace}
        n_prompt = {t.req_id: t.n_prompt for t in trace}
        for rec in recs:
            for rid, L, c in zip(rec.req_ids, rec.n_new, rec.n_ctx):
                if c < n_prompt[rid]:
                    assert c == prompt_done[rid]
                    prompt_done[rid] += L
                if c + L >= n_prompt[rid]:
                    gen[rid] += 1
        assert prompt_done == n_prompt
        assert all(gen[t.req_id] == t.out_len for t in trace)


# ---------------------------------------------------------------- paged K/V (CS349D Lecture 2, 5.1 and 6.1)

def test_block_pool_lowest_first_and_release():
    b = scheduler.BlockPool(5 * scheduler.KV_BLOCK)
    assert b.grow(7, 2) and b.table[7] == [0, 1]
    assert b.grow(8, 1) and b.table[8] == [2]
    assert not b.grow(9, 3) and b.held(9) == 0          # all or nothing
    b.release(7)
    assert b.grow(9, 3) and b.table[9] == [0, 1, 3]      # lowest free blocks first
    assert b.n_rsrv == 4 * scheduler.KV_BLOCK


def test_paged_with_ample_memory_is_algorithm_1():
    rng = np.random.default_rng(45)
    for trial in range(15):
        n = int(rng.integers(3, 25))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 60)), int(rng.integers(1, 12))
            trace.append(_R(i, int(rng.integers(0, 20)), lp, lo, lp + lo + int(rng.integers(0, 4))))
        kw = dict(max_bs=int(rng.integers(1, 9)))
        plain = scheduler.run_schedule(trace, n_slots=100_000, **kw)
        paged = scheduler.run_schedule(trace, n_slots=100_000 // 32 * 32, policy=scheduler.RESERVE_PAGED, **kw)
        assert _records(plain) == _records(paged)
        assert all(not r.preempted for r in paged)


def test_paged_preemption_by_hand():
    # two blocks (64 slots); A and B: prompt 30, 10 tokens each, both at 0.
    #  it 0-2: both fit in one block each (positions 0..31)
    #  it 3:   A's position 32 needs a second block; none is free, so the
    #          latest arrival holding blocks (B) is preempted; B then needs
    #          two blocks to recompute 33 known tokens and does not fit
    #  it 4-9: A alone; it finishes at it 9 and frees both blocks
    #  it 10:  B recomputes its 33 known tokens (30 prompt + 3 generated)
    trace = [_R(0, 0, 30, 10, 40), _R(1, 0, 30, 10, 40)]
    recs = scheduler.run_schedule(trace, max_bs=4, n_slots=64, policy=scheduler.RESERVE_PAGED)
    got = [(r.it, r.req_ids, r.n_new, r.n_ctx, sorted(r.released), r.preempted) for r in recs]
    want = [(0, [0, 1], [30, 30], [0, 0], [], []), (1, [0, 1], [1, 1], [30, 30], [], []),
            (2, [0, 1], [1, 1], [31, 31], [], []), (3, [0], [1], [32], [], [1])]
    want += [(t, [0], [1], [29 + t], [0] if t == 9 else [], []) for t in range(4, 10)]
    want += [(10, [1], [33], [0], [], [])]
    want += [(t, [1], [1], [22 + t], [1] if t == 16 else [], []) for t in range(11, 17)]
    assert got == want


def test_paged_invariants_random_traces():
    rng = np.random.default_rng(46)
    n_preempted = 0
    for trial in range(30):
        n = int(rng.integers(2, 20))
        trace = []
        for i in range(n):
            lp, lo = int(rng.integers(1, 70)), int(rng.integers(1, 40))
            trace.append(_R(i, int(rng.integers(0, 20)), lp, lo, lp + lo + int(rng.integers(0, 4))))
        need = max(-(-(t.n_prompt + t.out_len) // 32) for t in trace)
        n_slots = 32 * int(rng.integers(need, 2 * need + 3))
        kw = dict(max_bs=int(rng.integers(1, 9)), n_slots=n_slots, policy=scheduler.RESERVE_PAGED)
        if trial % 3 == 0:
            kw.update(token_budget=int(rng.integers(8, 64)), chunk=int(rng.integers(4, 40)))
        recs = scheduler.run_schedule(trace, **kw)
        gen = {t.req_id: 0 for t in trace}
        known = {t.req_id: t.n_prompt for t in trace}
        cached = {t.req_id: 0 for t in trace}
        for rec in recs:
            for rid in rec.preempted:
                cached[rid] = 0
                n_preempted += 1
            held = 0
            for rid, L, c in zip(rec.req_ids, rec.n_new, rec.n_ctx):
                assert c == cached[rid] and 1 <= L <= known[rid] - c
                cached[rid] += L
                if cached[rid] == known[rid]:
                    gen[rid] += 1
                    known[rid] += 1
                held += -(-cached[rid] // 32)
            assert held * 32 <= n_slots
        assert all(gen[t.req_id] == t.out_len for t in trace)
    assert n_preempted > 0   # the traces do exercise preemption

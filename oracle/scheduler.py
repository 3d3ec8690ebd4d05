"""Iteration-level FCFS scheduling (Orca Algorithm 1) with n_workers = 1.

Algorithm 1 ("ORCA scheduling algorithm", Orca walk-through, section
"两个约束：max batch size 与 GPU 显存"): Select drops RUNNING requests, sorts
the rest by arrival, takes at most max_bs of them, and reserves max_tokens
K/V slots for each INITIATION request; when a reservation would exceed
n_slots it stops selecting (break, never skip: skipping would break FCFS).
The main loop marks the batch RUNNING, runs one iteration, marks the
returned requests INCREMENT and releases max_tokens for finished ones.

Readings where the extracted text is garbled:
* the per-request batch insertion applies to every non-RUNNING request,
  INCREMENT included (the notes' select_batch sketch appends every request;
  the walk-through's indentation puts it inside the INITIATION branch);
* with one worker each batch returns before the next Select;
* ties in arrival are broken by request id;
* a request is finished when it has generated out_len tokens (no EOS, per
  the evaluation setup) or prompt + generated >= max_tokens;
* the slot pool gives each request one contiguous segment, first fit at the
  lowest base; a reservation that passes the count rule but finds no hole
  fails like a count failure (break).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

INITIATION, INCREMENT, RUNNING, FINISHED = 0, 1, 2, 3


class SlotPool:
    """Contiguous K/V slot reservations over [0, n_slots)."""

    def __init__(self, n_slots: int):
        self.n_slots = n_slots
        self.n_rsrv = 0
        self.free: List[Tuple[int, int]] = [(0, n_slots)] if n_slots > 0 else []  # (base, length)
        self.owned: Dict[int, Tuple[int, int]] = {}
        self.frag_blocks = 0

    def reserve(self, req_id: int, n: int) -> Optional[int]:
        if n <= 0 or req_id in self.owned:
            raise ValueError("invalid reservation")
        if self.n_rsrv + n > self.n_slots:
            return None
        for i, (base, length) in enumerate(self.free):
            if length >= n:
                if length == n:
                    del self.free[i]
                else:
                    self.free[i] = (base + n, length - n)
                self.owned[req_id] = (base, n)
                self.n_rsrv += n
                return base
        self.frag_blocks += 1
        return None

    def release(self, req_id: int) -> None:
        if req_id not in self.owned:
            raise KeyError(req_id)
        base, n = self.owned.pop(req_id)
        self.n_rsrv -= n
        self.free.append((base, n))
        self.free.sort()
        merged: List[Tuple[int, int]] = []
        for b, l in self.free:
            if merged and merged[-1][0] + merged[-1][1] == b:
                merged[-1] = (merged[-1][0], merged[-1][1] + l)
            else:
                merged.append((b, l))
        self.free = merged


@dataclasses.dataclass
class ReqState:
    req_id: int
    arrival: int
    n_prompt: int
    out_len: int
    max_tokens: int
    state: int = INITIATION
    n_cached: int = 0
    n_generated: int = 0
    slot_base: int = -1
    preempted: int = 0


RESERVE_MAX, RESERVE_POW2, RESERVE_ORACLE, RESERVE_PAGED = 0, 1, 2, 3
KV_BLOCK = 32


class BlockPool:
    """Paged K/V (CS349D Lecture 2, sections 5.1 and 6.1: memory handed out
    block by block as requests grow, nothing reserved ahead): n_slots //
    KV_BLOCK blocks; each request holds a list of blocks in position order;
    the lowest free block is handed out first."""

    def __init__(self, n_slots: int):
        self.n_slots = n_slots
        self.n_blocks = n_slots // KV_BLOCK
        self.free = list(range(self.n_blocks))   # kept sorted
        self.table: Dict[int, List[int]] = {}

    @property
    def n_rsrv(self) -> int:   # slots held
        return (self.n_blocks - len(self.free)) * KV_BLOCK

    def held(self, req_id: int) -> int:
        return len(self.table.get(req_id, []))

    def grow(self, req_id: int, total: int) -> bool:
        need = total - self.held(req_id)
        if need <= 0:
            return True
        if len(self.free) < need:
            return False
        t = self.table.setdefault(req_id, [])
        t.extend(self.free[:need])
        del self.free[:need]
        return True

    def release(self, req_id: int) -> None:
        blocks = self.table.pop(req_id)
        self.free = sorted(self.free + blocks)


def reserve_size(policy: int, r: ReqState) -> int:
    """Slots a request reserves at first schedule (CS349D Lecture 2, section
    6.1, the three ways Orca is re-implemented there): Max reserves
    max_tokens, the most the request may reach; Pow2 reserves its true
    final length (prompt + output) rounded up to a power of two, as with an
    imprecise length prediction; Oracle reserves exactly the true final
    length.  Reading: "true final length" is n_prompt + out_len, capped at
    max_tokens (a request never grows past max_tokens), and so are the other
    two."""
    true_len = min(r.n_prompt + r.out_len, r.max_tokens)
    if policy == RESERVE_ORACLE:
        return true_len
    if policy == RESERVE_POW2:
        p = 1
        while p < true_len:
            p *= 2
        return min(p, r.max_tokens)
    return r.max_tokens


def preempt(r: ReqState, blocks: BlockPool) -> None:
    """Free the request's blocks; it recomputes its known tokens when it is
    selected again (CS349D Lecture 2, section 5.1: the latest arrival is
    kicked out and recomputed later)."""
    blocks.release(r.req_id)
    r.n_cached = 0
    r.state = INITIATION
    r.preempted += 1


def select(pool: List[ReqState], slots, max_bs: int, policy: int = RESERVE_MAX,
           chunk: Optional[int] = None) -> List[ReqState]:
    """Algorithm 1 Select over the arrived, unfinished requests.

    Paged K/V (slots is a BlockPool): the same walk grows each candidate's
    block table to cover the rows it runs this iteration (the rest of its
    known tokens, at most `chunk`).  When the pool is short, the latest
    arrivals holding blocks that are not in the batch (and not running) are
    preempted; if that is not enough, a candidate holding no blocks ends the
    selection (as a failed reservation does) and one holding blocks is
    itself preempted and ends it.  Readings: "latest arrival" is the largest
    (arrival, request id); preempted requests recompute from position 0."""
    cands = sorted((r for r in pool if r.state in (INITIATION, INCREMENT)),
                   key=lambda r: (r.arrival, r.req_id))
    batch: List[ReqState] = []
    for r in cands:
        if len(batch) == max_bs:
            break
        if policy == RESERVE_PAGED:
            rows = min(default_rows(r), chunk) if chunk else default_rows(r)
            total = -(-(r.n_cached + rows) // KV_BLOCK)
            while len(slots.free) < total - slots.held(r.req_id):
                victims = [q for q in pool if q is not r and q not in batch and q.state == INCREMENT
                           and slots.held(q.req_id) > 0]
                if not victims:
                    break
                preempt(max(victims, key=lambda q: (q.arrival, q.req_id)), slots)
            if not slots.grow(r.req_id, total):
                if slots.held(r.req_id) > 0:
                    preempt(r, slots)
                break
            r.state = INCREMENT
            batch.append(r)
            continue
        if r.state == INITIATION:
            base = slots.reserve(r.req_id, reserve_size(policy, r))
            if base is None:
                break
            r.slot_base = base
        batch.append(r)
    return batch


def kv_usage(pool: List[ReqState], slots: SlotPool) -> Tuple[int, int]:
    """(reserved slots, slots holding K/V): CS349D Lecture 2, section 6.1
    contrasts the memory a reservation occupies with what is written."""
    if isinstance(slots, BlockPool):
        stored = sum(r.n_cached for r in pool if r.state not in (INITIATION, FINISHED) and slots.held(r.req_id))
    else:
        stored = sum(r.n_cached for r in pool if r.state not in (INITIATION, FINISHED) and r.slot_base >= 0)
    return slots.n_rsrv, stored


def known_len(r: ReqState) -> int:
    """Tokens of the request known so far: prompt + generated."""
    return r.n_prompt + r.n_generated


def default_rows(r: ReqState) -> int:
    """Rows of a selected request: its known tokens not yet in the K/V
    slots - the rest of its prompt (all of it at first schedule), one decode
    row, or, after a preemption, the prompt and the generated tokens again."""
    return max(1, known_len(r) - r.n_cached)


def decoding(r: ReqState) -> bool:
    return r.n_generated > 0 and r.n_cached == known_len(r) - 1


def select_budget(pool: List[ReqState], slots: SlotPool, max_bs: int, token_budget: int,
                  chunk: int, policy: int = RESERVE_MAX) -> List[Tuple[ReqState, int]]:
    """Chunked prefill under a per-iteration token budget, on top of
    Algorithm 1.

    CS349D Lecture 2, Exercise 9: cut long prompts into chunks, mix chunks
    into the iterations and cap the tokens of one iteration; the engine then
    runs SeqWork(n_new = chunk, n_past = prompt tokens already processed).
    Static-to-continuous article, chunked prefill: decode first, the rest of
    the budget goes to prompt chunks.  Reading: Algorithm 1 Select is kept
    as it is (FCFS, max_bs, reservation at first schedule, break); over the
    selected requests, in batch order, every decoding request takes one row
    while the budget lasts, then every prompting request takes
    min(remaining prompt, chunk, budget left) rows.  Returns (request, rows)
    in batch order; rows may be 0 (admitted but idle this iteration)."""
    batch = select(pool, slots, max_bs, policy, chunk)
    left = token_budget
    rows: Dict[int, int] = {}
    for r in batch:
        if decoding(r) and left >= 1:
            rows[r.req_id] = 1
            left -= 1
    for r in batch:
        if not decoding(r):
            n = min(default_rows(r), chunk, left)
            rows[r.req_id] = n
            left -= n
    return [(r, rows.get(r.req_id, 0)) for r in batch]


def finished(r: ReqState) -> bool:
    return r.n_generated >= r.out_len or r.n_prompt + r.n_generated >= r.max_tokens


@dataclasses.dataclass
class IterRecord:
    it: int
    req_ids: List[int]
    n_new: List[int]        # L_i: prompt length for a prefill, 1 for a decode
    n_ctx: List[int]        # c_i: tokens cached before this iteration
    slot_base: List[int]
    released: List[int]
    preempted: List[int] = dataclasses.field(default_factory=list)
    # (reserved, stored) K/V slots once this iteration's results are applied
    kv: Tuple[int, int] = (0, 0)


def run_schedule(trace, max_bs: int, n_slots: int, max_iters: int = 10_000_000,
                 token_budget: Optional[int] = None, chunk: Optional[int] = None,
                 policy: int = RESERVE_MAX, n_workers: int = 1) -> List[IterRecord]:
    """Drive Algorithm 1 over a trace whose arrivals are iteration indices.

    A request whose arrival is t can be selected at iteration t.  When no
    request is in the pool the clock jumps to the next arrival (no iteration
    is run).  Raises RuntimeError if the pool is non-empty but nothing can
    ever be selected (a head request larger than n_slots).  With a token
    budget or a chunk size the batch comes from select_budget: a prompt
    chunk that leaves part of the prompt unprocessed generates no token.

    n_workers: batches kept scheduled at once (Algorithm 1's main loop:
    select and schedule a batch, count it, and once n_workers batches are
    scheduled wait for the oldest to return before selecting again).  The
    requests of a scheduled batch are RUNNING, so the next Select skips
    them.  Readings: the clock counts scheduled batches; a Select that finds
    nothing to run does not schedule an empty batch, it waits for the
    oldest batch in flight instead (or, with none in flight, the clock jumps
    to the next arrival).  Records are in scheduling order."""
    order = sorted(trace, key=lambda r: (r.arrival, r.req_id))
    states = [ReqState(r.req_id, r.arrival, r.n_prompt, r.out_len, r.max_tokens) for r in order]
    slots = BlockPool(n_slots) if policy == RESERVE_PAGED else SlotPool(n_slots)
    pool: List[ReqState] = []
    nxt = 0
    it = 0
    records: List[IterRecord] = []
    inflight: List[Tuple[IterRecord, List[Tuple[ReqState, int]]]] = []
    budgeted = token_budget is not None or chunk is not None
    big = 2 ** 31 - 1
    while nxt < len(states) or pool:
        while nxt < len(states) and states[nxt].arrival <= it:
            pool.append(states[nxt])
            nxt += 1
        before = {r.req_id: r.preempted for r in pool}
        if budgeted:
            sel = select_budget(pool, slots, max_bs, token_budget or big, chunk or big, policy)
        else:
            sel = [(r, default_rows(r)) for r in select(pool, slots, max_bs, policy)]
        preempted = sorted(r.req_id for r in pool if r.preempted != before[r.req_id])
        run = [(r, n) for r, n in sel if n > 0]
        for r, n in sel:
            if n == 0:
                r.state = INCREMENT  # admitted (slots reserved) but idle this iteration
        if run:
            rec = IterRecord(it, [r.req_id for r, _ in run], [n for _, n in run], [r.n_cached for r, _ in run],
                             [r.slot_base for r, _ in run], [], preempted)
            for r, _ in run:
                r.state = RUNNING
            inflight.append((rec, run))
            records.append(rec)
            it += 1
            if len(records) > max_iters:
                raise RuntimeError("iteration limit")
        if inflight and (len(inflight) == n_workers or not run):
            rec, done_run = inflight.pop(0)
            for r, n in done_run:
                r.state = INCREMENT
                r.n_cached += n
                if r.n_cached < known_len(r):
                    continue  # a chunk: known tokens remain unprocessed, nothing generated yet
                r.n_generated += 1
                if finished(r):
                    r.state = FINISHED
                    slots.release(r.req_id)
                    rec.released.append(r.req_id)
            pool = [r for r in pool if r.state != FINISHED]
            rec.kv = kv_usage(states, slots)
        elif not run:
            if pool:
                raise RuntimeError(f"no request can be scheduled at iteration {it}")
            it = states[nxt].arrival  # idle: the clock jumps to the next arrival
    return records

"""PyTorch plumbing around liborca: device memory, streams, the request pool
and the iteration-level serving loop.

PyTorch only allocates device memory and provides the stream; every kernel
of the iteration runs in liborca.  The serving loop follows Algorithm 1 with
one worker (Orca walk-through, Algorithm 1): each iteration admits the
requests that have arrived, calls orca_select_batch, then orca_iteration,
which also applies the post-iteration state updates and releases the slots
of finished requests.
"""
from __future__ import annotations

import ctypes
import dataclasses
import time
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import _orca as C

LAYER_TENSORS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                 "ln2_g", "ln2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2")
GLOBAL_TENSORS = ("tok_emb", "pos_emb", "lnf_g", "lnf_b")


def _is_matrix(name: str) -> bool:
    return name.startswith("w_") or name.endswith("_emb")


RESERVE_POLICIES = {"max": C.ORCA_RESERVE_MAX, "pow2": C.ORCA_RESERVE_POW2, "oracle": C.ORCA_RESERVE_ORACLE,
                    "paged": C.ORCA_RESERVE_PAGED}


def make_config(shape, max_bs: int, n_slots: int, max_rows: int, reserve_policy: int = C.ORCA_RESERVE_MAX
                ) -> C.orca_config:
    return C.orca_config(n_layers=shape.n_layers, hidden=shape.hidden, n_heads=shape.n_heads, ffn=shape.ffn,
                         vocab=shape.vocab, max_pos=shape.max_pos, dtype=shape.dtype, max_bs=max_bs,
                         n_slots=n_slots, max_rows=max_rows, reserve_policy=reserve_policy)


class DeviceWeights:
    """Weights on the device in the order orca_engine_create expects.

    `host` maps names ("tok_emb", "L0.w_qkv", ...) to fp32 numpy arrays whose
    values are exact in the model dtype; `generator` instead draws N(0, std)
    matrices on the device (for shapes too large to build on the host)."""

    def __init__(self, shape, device, host: Optional[Dict[str, np.ndarray]] = None, seed: int = 0,
                 w_std: float = 0.02):
        self.shape = shape
        mdt = torch.bfloat16 if shape.dtype == C.ORCA_DTYPE_BF16 else torch.float32
        H, F, V, P = shape.hidden, shape.ffn, shape.vocab, shape.max_pos
        shapes = {"tok_emb": (V, H), "pos_emb": (P, H), "lnf_g": (H,), "lnf_b": (H,),
                  "ln1_g": (H,), "ln1_b": (H,), "w_qkv": (3 * H, H), "b_qkv": (3 * H,), "w_o": (H, H),
                  "b_o": (H,), "ln2_g": (H,), "ln2_b": (H,), "w_fc1": (F, H), "b_fc1": (F,),
                  "w_fc2": (H, F), "b_fc2": (H,)}
        gen = None
        if host is None:
            gen = torch.Generator(device=device)
            gen.manual_seed(seed)
        self.tensors: List[torch.Tensor] = []
        names = list(GLOBAL_TENSORS) + [f"L{l}.{n}" for l in range(shape.n_layers) for n in LAYER_TENSORS]
        for full in names:
            base = full.split(".", 1)[-1]
            dt = mdt if _is_matrix(base) else torch.float32
            if host is not None:
                t = torch.from_numpy(np.ascontiguousarray(host[full], dtype=np.float32)).to(device=device, dtype=dt)
            elif _is_matrix(base):
                t = (torch.randn(shapes[base], device=device, generator=gen) * w_std).to(dt)
            elif base.endswith("_g"):
                t = torch.ones(shapes[base], device=device, dtype=dt)
            else:
                t = torch.zeros(shapes[base], device=device, dtype=dt)
            self.tensors.append(t.contiguous())
        self.ptrs = [t.data_ptr() for t in self.tensors]

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.tensors)


class Engine:
    """liborca engine with torch-allocated K/V pool and workspace."""

    def __init__(self, shape, weights: DeviceWeights, max_bs: int, n_slots: int, max_rows: int, device=None,
                 reserve_policy: int = C.ORCA_RESERVE_MAX):
        self.shape = shape
        self.device = torch.device(device if device is not None else "cuda")
        self.cfg = make_config(shape, max_bs, n_slots, max_rows, reserve_policy)
        self.kv_bytes = C.orca_kv_pool_bytes(self.cfg)
        self.ws_bytes = C.orca_workspace_bytes(self.cfg)
        self.kv = torch.empty(self.kv_bytes, dtype=torch.uint8, device=self.device)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.weights = weights
        with torch.cuda.device(self.device):
            self.handle = C.orca_engine_create(self.cfg, weights.ptrs, self.kv.data_ptr(), self.kv_bytes,
                                               self.ws.data_ptr(), self.ws_bytes)
        self.max_bs = max_bs

    def kv_view(self) -> torch.Tensor:
        """The K/V pool as [n_layers, 2, n_heads, n_slots, head_dim] (model dtype)."""
        s = self.shape
        dt = torch.bfloat16 if s.dtype == C.ORCA_DTYPE_BF16 else torch.float32
        return self.kv.view(dt).view(s.n_layers, 2, s.n_heads, self.cfg.n_slots, s.hidden // s.n_heads)

    def close(self):
        if getattr(self, "handle", None):
            C.orca_engine_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# numpy view of orca_request (same layout as the C struct)
REQUEST_DTYPE = np.dtype([("req_id", "<i8"), ("arrival", "<i8"), ("state", "<i4"), ("n_prompt", "<i4"),
                          ("max_tokens", "<i4"), ("out_len", "<i4"), ("n_cached", "<i4"), ("n_generated", "<i4"),
                          ("n_sched", "<i4"), ("n_reserved", "<i4"), ("slot_base", "<i8"), ("tokens", "<u8")])
assert REQUEST_DTYPE.itemsize == ctypes.sizeof(C.orca_request)


class RequestPool:
    """ctypes array of orca_request with numpy token buffers, in arrival order."""

    def __init__(self, requests: Sequence, teacher_force: bool = False):
        reqs = sorted(requests, key=lambda r: (r.arrival, r.req_id))
        self.reqs = reqs
        self.n = len(reqs)
        self.arr = (C.orca_request * max(1, self.n))()
        self.tokens: List[np.ndarray] = []
        for i, r in enumerate(reqs):
            buf = np.zeros(r.n_prompt + r.out_len, dtype=np.int32)
            buf[:r.n_prompt] = r.prompt
            if teacher_force:
                if r.forced is None:
                    raise ValueError("teacher forcing needs forced continuations")
                buf[r.n_prompt:] = r.forced[:r.out_len]
            self.tokens.append(buf)
            self.arr[i] = C.orca_request(req_id=r.req_id, arrival=r.arrival, state=C.ORCA_INITIATION,
                                         n_prompt=r.n_prompt, max_tokens=r.max_tokens, out_len=r.out_len,
                                         n_cached=0, n_generated=0, slot_base=-1,
                                         tokens=buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
        self.view = np.frombuffer(self.arr, dtype=REQUEST_DTYPE)   # shares memory with arr
        self.arrivals = np.array([r.arrival for r in reqs], dtype=np.int64)

    def reset(self):
        for i, r in enumerate(self.reqs):
            a = self.arr[i]
            a.state, a.n_cached, a.n_generated, a.slot_base = C.ORCA_INITIATION, 0, 0, -1
            a.n_sched, a.n_reserved = 0, 0


@dataclasses.dataclass
class IterRecord:
    it: int
    req_ids: List[int]
    n_new: List[int]
    n_ctx: List[int]
    slot_base: List[int]
    released: List[int]
    next_tokens: List[int]
    logits: Optional[np.ndarray] = None
    launches: int = 0          # kernels the iteration launched on the device
    preempted: List[int] = dataclasses.field(default_factory=list)  # paged K/V: requests sent back by this Select
    kv: Optional[tuple] = None  # (reserved, stored) K/V slots after the iteration (track_kv)


class ServingLoop:
    """Iteration-level scheduling over a RequestPool (Algorithm 1).

    Arrivals are iteration indices: a request whose arrival is t can be
    selected at iteration t.  n_workers batches may be scheduled at once
    (Algorithm 1's main loop; on one GPU the host selects and enqueues the
    next batch while the previous one runs): the requests of a batch in
    flight are RUNNING and the next Select skips them; once n_workers
    batches are in flight, or when nothing else can be selected, the oldest
    is waited for.  When nothing has arrived the clock jumps to the next
    arrival.  step() returns the record of the next iteration to complete,
    in scheduling order."""

    def __init__(self, engine: Engine, pool: RequestPool, teacher_force: bool = False, keep_logits: bool = False,
                 stream: Optional[torch.cuda.Stream] = None, keep_ids: Optional[set] = None, eager: bool = False,
                 token_budget: Optional[int] = None, chunk: Optional[int] = None, n_workers: int = 1,
                 track_kv: bool = False):
        if n_workers not in (1, 2):
            raise ValueError("n_workers must be 1 or 2")
        self.eng, self.pool = engine, pool
        self.n_workers = n_workers
        self.track_kv = track_kv
        self.flags = (C.ORCA_ITER_TEACHER_FORCE if teacher_force else 0) | (C.ORCA_ITER_EAGER if eager else 0)
        keep_logits = keep_logits or keep_ids is not None
        self.keep_logits = keep_logits
        self.keep_ids = keep_ids
        self.stream = stream if stream is not None else torch.cuda.current_stream(engine.device)
        self.batch_idx = (ctypes.c_int32 * engine.max_bs)()
        self.next_tok = (ctypes.c_int32 * engine.max_bs)()
        self._bi = np.frombuffer(self.batch_idx, dtype=np.int32)
        self._nt = np.frombuffer(self.next_tok, dtype=np.int32)
        # one logits buffer per iteration that can be in flight
        self.logits = ([torch.empty((engine.max_bs, engine.shape.vocab), dtype=torch.float32, device=engine.device)
                        for _ in range(n_workers)] if keep_logits else None)
        # chunked prefill under a per-iteration token budget (None: plain Algorithm 1)
        self.budget = None
        if token_budget is not None or chunk is not None:
            big = 2 ** 31 - 1
            self.budget = (token_budget or big, chunk or big)
        self.it = 0
        self.n_arrived = 0
        self.n_done = 0
        self.n_submitted = 0
        self.inflight: List[tuple] = []   # (record, pool indices, logits buffer), oldest first
        self.preempted: List[int] = []    # preemptions not yet attached to a record
        # host seconds spent selecting / submitting / completing (diagnostics)
        self.t_pre = self.t_call = self.t_post = 0.0

    def done(self) -> bool:
        return self.n_done >= self.pool.n and not self.inflight

    def _complete(self) -> IterRecord:
        t0 = time.perf_counter()
        rec, idx, lg = self.inflight.pop(0)
        nb = C.orca_iteration_wait(self.eng.handle, self.batch_idx, self.next_tok)
        t1 = time.perf_counter()
        rec.next_tokens = self._nt[:nb].tolist()
        P = self.pool
        done = P.view["state"][idx] == C.ORCA_FINISHED
        if done.any():
            rec.released = P.view["req_id"][idx][done].tolist()
            self.n_done += int(done.sum())
        if self.track_kv:
            rec.kv = C.orca_kv_usage(self.eng.handle, P.arr, self.n_arrived)
        if lg is not None:
            if self.keep_ids is None:
                rec.logits = lg[:nb].cpu().numpy()
            else:
                rows = [k for k, rid in enumerate(rec.req_ids) if rid in self.keep_ids]
                if rows:
                    sel_l = lg[torch.tensor(rows, device=lg.device)].cpu().numpy()
                    rec.logits = {rec.req_ids[k]: sel_l[j] for j, k in enumerate(rows)}
        self.t_call += t1 - t0
        self.t_post += time.perf_counter() - t1
        return rec

    def step(self) -> Optional[IterRecord]:
        P = self.pool
        while True:
            t0 = time.perf_counter()
            if self.n_arrived < P.n and P.arrivals[self.n_arrived] <= self.it:
                self.n_arrived = int(np.searchsorted(P.arrivals, self.it, side="right"))
            held = P.view["state"][:self.n_arrived] == C.ORCA_INCREMENT
            if self.budget is None:
                nb = C.orca_select_batch(self.eng.handle, P.arr, self.n_arrived, self.batch_idx)
            else:
                nb = C.orca_select_batch_budget(self.eng.handle, P.arr, self.n_arrived, self.budget[0],
                                                self.budget[1], self.batch_idx)
            gone = held & (P.view["state"][:self.n_arrived] == C.ORCA_INITIATION)   # preempted (paged K/V)
            if gone.any():
                self.preempted += sorted(P.view["req_id"][:self.n_arrived][gone].tolist())
            if nb > 0:
                idx = self._bi[:nb].copy()
                sel = P.view[idx]
                rec = IterRecord(self.it, sel["req_id"].tolist(), sel["n_sched"].tolist(), sel["n_cached"].tolist(),
                                 sel["slot_base"].tolist(), [], [], preempted=sorted(self.preempted))
                self.preempted = []
                lg = self.logits[self.n_submitted % self.n_workers] if self.logits is not None else None
                t1 = time.perf_counter()
                C.orca_iteration_submit(self.eng.handle, P.arr, self.batch_idx, nb, self.flags,
                                        lg.data_ptr() if lg is not None else 0, self.stream.cuda_stream)
                rec.launches = C.orca_last_launches(self.eng.handle)
                self.inflight.append((rec, idx, lg))
                self.n_submitted += 1
                self.it += 1
                self.t_pre += t1 - t0
                self.t_call += time.perf_counter() - t1
            if self.inflight and (len(self.inflight) == self.n_workers or nb == 0):
                return self._complete()
            if nb == 0:
                if self.n_arrived - self.n_done == 0 and self.n_arrived < P.n:
                    self.it = int(P.arrivals[self.n_arrived])   # idle: jump to the next arrival
                    continue
                raise RuntimeError(f"no request can be scheduled at iteration {self.it}")

    def run(self, max_iters: int = 10_000_000) -> List[IterRecord]:
        recs = []
        while not self.done() and len(recs) < max_iters:
            recs.append(self.step())
        return recs

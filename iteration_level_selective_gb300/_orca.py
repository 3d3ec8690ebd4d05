"""ctypes binding of liborca (include/orca.h): same names, argument marshalling only.

Every step of the iteration runs inside liborca's CUDA kernels; this module
only converts Python arguments to the C types and raises OrcaError on a
non-zero return code.  If liborca.so has not been built the import of the
library fails loudly: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liborca.so")

ORCA_OK = 0
ORCA_EINVAL = -1
ORCA_ENOSLOTS = -2
ORCA_EBATCH = -3
ORCA_EUNKNOWN_REQ = -4
ORCA_EDOUBLE_RELEASE = -5
ORCA_EDEVICE = -6
ORCA_ECUDA = -7
ORCA_ESTATE = -8
ERROR_NAMES = {ORCA_EINVAL: "EINVAL", ORCA_ENOSLOTS: "ENOSLOTS", ORCA_EBATCH: "EBATCH",
               ORCA_EUNKNOWN_REQ: "EUNKNOWN_REQ", ORCA_EDOUBLE_RELEASE: "EDOUBLE_RELEASE",
               ORCA_EDEVICE: "EDEVICE", ORCA_ECUDA: "ECUDA", ORCA_ESTATE: "ESTATE"}

ORCA_DTYPE_F32 = 0
ORCA_DTYPE_BF16 = 1
ORCA_INITIATION, ORCA_INCREMENT, ORCA_RUNNING, ORCA_FINISHED = 0, 1, 2, 3
ORCA_RESERVE_MAX, ORCA_RESERVE_POW2, ORCA_RESERVE_ORACLE, ORCA_RESERVE_PAGED = 0, 1, 2, 3
ORCA_KV_BLOCK = 32
ORCA_ITER_TEACHER_FORCE = 1
ORCA_ITER_EAGER = 2
ORCA_ITER_SELFTEST_TIMEOUT = 4
(ORCA_K_EMBED, ORCA_K_LAYERNORM, ORCA_K_GEMM_QKV, ORCA_K_ATTENTION, ORCA_K_GEMM_O, ORCA_K_GEMM_FC1,
 ORCA_K_GEMM_FC2, ORCA_K_LM_HEAD, ORCA_K_ARGMAX, ORCA_K_COUNT) = range(10)
KERNEL_NAMES = ["embed", "layernorm", "gemm_qkv", "attention", "gemm_o", "gemm_fc1", "gemm_fc2",
                "lm_head", "argmax"]


class OrcaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class orca_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("vocab", ctypes.c_int32), ("max_pos", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("max_bs", ctypes.c_int32), ("n_slots", ctypes.c_int64),
                ("max_rows", ctypes.c_int32), ("reserve_policy", ctypes.c_int32)]


class orca_request(ctypes.Structure):
    _fields_ = [("req_id", ctypes.c_int64), ("arrival", ctypes.c_int64), ("state", ctypes.c_int32),
                ("n_prompt", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("out_len", ctypes.c_int32),
                ("n_cached", ctypes.c_int32), ("n_generated", ctypes.c_int32), ("n_sched", ctypes.c_int32),
                ("n_reserved", ctypes.c_int32), ("slot_base", ctypes.c_int64),
                ("tokens", ctypes.POINTER(ctypes.c_int32))]


class orca_kernel_stats(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64), ("total_ms", ctypes.c_double), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double)]


class orca_gemm_plan_info(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("tiles", ctypes.c_int32), ("k_split", ctypes.c_int32), ("ranges", ctypes.c_int32),
                ("workers", ctypes.c_int32), ("code", ctypes.c_int32)]


EXPORTS = ("orca_kv_pool_bytes", "orca_workspace_bytes", "orca_weight_count", "orca_engine_create",
           "orca_engine_destroy", "orca_kv_reserve", "orca_kv_release", "orca_kv_stats", "orca_select_batch",
           "orca_iteration", "orca_last_descriptor", "orca_argmax_rows", "orca_profile_enable",
           "orca_profile_read", "orca_last_error", "orca_linear", "orca_last_transfer",
           "orca_attention_workspace_bytes", "orca_attention", "orca_attention_noalloc", "orca_last_launches",
           "orca_select_batch_budget", "orca_kv_usage", "orca_iteration_submit", "orca_iteration_wait",
           "orca_selftest_wait_timeout", "orca_gemm_plan_query", "orca_gemm_pair_segments")

_lib = None


def lib() -> ctypes.CDLL:
    """Load liborca.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with iteration_level_selective_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, c_i32, c_i64, c_sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(orca_config)
        reqp = ctypes.POINTER(orca_request)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        sig = {
            "orca_kv_pool_bytes": [cfgp, ctypes.POINTER(c_sz)],
            "orca_workspace_bytes": [cfgp, ctypes.POINTER(c_sz)],
            "orca_weight_count": [cfgp, i32p],
            "orca_engine_create": [cfgp, ctypes.POINTER(P), c_i32, P, c_sz, P, c_sz, ctypes.POINTER(P)],
            "orca_engine_destroy": [P],
            "orca_kv_reserve": [P, c_i64, c_i32, i64p],
            "orca_kv_release": [P, c_i64],
            "orca_kv_stats": [P, i64p, i64p, i64p],
            "orca_kv_usage": [P, reqp, c_i32, i64p, i64p],
            "orca_select_batch": [P, reqp, c_i32, i32p, i32p],
            "orca_select_batch_budget": [P, reqp, c_i32, c_i32, c_i32, i32p, i32p],
            "orca_iteration": [P, reqp, i32p, c_i32, c_i32, i32p, P, P],
            "orca_iteration_submit": [P, reqp, i32p, c_i32, c_i32, P, P],
            "orca_iteration_wait": [P, i32p, i32p, i32p],
            "orca_last_descriptor": [P, i32p, i32p, i32p, i32p, i32p, i32p, c_i32],
            "orca_argmax_rows": [P, c_i32, c_i32, P, P],
            "orca_profile_enable": [P, c_i32],
            "orca_profile_read": [P, c_i32, ctypes.POINTER(orca_kernel_stats)],
            "orca_last_error": [P, ctypes.c_char_p, c_sz],
            "orca_linear": [c_i32, c_i32, P, P, P, P, c_i32, c_i32, c_i32, P, c_sz, P, P, P],
            "orca_last_transfer": [P, i64p, i64p, i32p],
            "orca_last_launches": [P, i32p],
            "orca_attention_workspace_bytes": [c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)],
            "orca_attention": [c_i32, c_i32, c_i32, c_i64, P, P, P, P, c_i32, i32p, i32p, i64p, P, c_sz, P, P],
            "orca_attention_noalloc": [c_i32, c_i32, c_i32, c_i64, P, P, P, P, c_i32, i32p, i32p, i64p, P, P],
            "orca_selftest_wait_timeout": [P, P],
            "orca_gemm_plan_query": [c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(orca_gemm_plan_info)],
            "orca_gemm_pair_segments": [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, i32p, c_i32],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int, eng=None) -> None:
    if rc != ORCA_OK:
        msg = ""
        if eng:
            buf = ctypes.create_string_buffer(512)
            lib().orca_last_error(eng, buf, 512)
            msg = buf.value.decode(errors="replace")
        raise OrcaError(rc, msg)


def orca_kv_pool_bytes(cfg: orca_config) -> int:
    n = ctypes.c_size_t()
    _check(lib().orca_kv_pool_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def orca_workspace_bytes(cfg: orca_config) -> int:
    n = ctypes.c_size_t()
    _check(lib().orca_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def orca_weight_count(cfg: orca_config) -> int:
    n = ctypes.c_int32()
    _check(lib().orca_weight_count(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def orca_engine_create(cfg: orca_config, weight_ptrs=None, kv_ptr=0, kv_bytes=0, ws_ptr=0, ws_bytes=0):
    """Returns an opaque engine handle (c_void_p).  weight_ptrs=None with
    kv_ptr = ws_ptr = 0 creates a host-only engine."""
    out = ctypes.c_void_p()
    if weight_ptrs is None:
        arr, n = None, 0
    else:
        arr = (ctypes.c_void_p * len(weight_ptrs))(*weight_ptrs)
        n = len(weight_ptrs)
    _check(lib().orca_engine_create(ctypes.byref(cfg), arr, n, ctypes.c_void_p(kv_ptr or None), kv_bytes,
                                    ctypes.c_void_p(ws_ptr or None), ws_bytes, ctypes.byref(out)))
    return out


def orca_engine_destroy(eng) -> None:
    _check(lib().orca_engine_destroy(eng))


def orca_kv_reserve(eng, req_id: int, n_tokens: int) -> int:
    base = ctypes.c_int64()
    _check(lib().orca_kv_reserve(eng, req_id, n_tokens, ctypes.byref(base)), eng)
    return base.value


def orca_kv_release(eng, req_id: int) -> None:
    _check(lib().orca_kv_release(eng, req_id), eng)


def orca_kv_stats(eng):
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().orca_kv_stats(eng, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), eng)
    return a.value, b.value, c.value


def orca_kv_usage(eng, pool, n_pool: int):
    """(reserved slots, slots holding K/V) over the pool."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().orca_kv_usage(eng, pool, n_pool, ctypes.byref(a), ctypes.byref(b)), eng)
    return a.value, b.value


def orca_select_batch(eng, pool, n_pool: int, batch_idx) -> int:
    """pool: ctypes array of orca_request; batch_idx: ctypes int32 array
    (capacity max_bs).  Returns n_batch."""
    nb = ctypes.c_int32()
    _check(lib().orca_select_batch(eng, pool, n_pool, batch_idx, ctypes.byref(nb)), eng)
    return nb.value


def orca_select_batch_budget(eng, pool, n_pool: int, token_budget: int, chunk: int, batch_idx) -> int:
    n = ctypes.c_int32()
    _check(lib().orca_select_batch_budget(eng, pool, n_pool, token_budget, chunk, batch_idx, ctypes.byref(n)), eng)
    return n.value


def orca_iteration(eng, pool, batch_idx, n_batch: int, flags: int, next_tokens, logits_ptr=0, stream=0) -> None:
    _check(lib().orca_iteration(eng, pool, batch_idx, n_batch, flags, next_tokens,
                                ctypes.c_void_p(logits_ptr or None), ctypes.c_void_p(stream or None)), eng)


def orca_iteration_submit(eng, pool, batch_idx, n_batch: int, flags: int, logits_ptr=0, stream=0) -> None:
    _check(lib().orca_iteration_submit(eng, pool, batch_idx, n_batch, flags, ctypes.c_void_p(logits_ptr or None),
                                       ctypes.c_void_p(stream or None)), eng)


def orca_iteration_wait(eng, batch_idx, next_tokens) -> int:
    """Wait for the oldest iteration in flight; returns its batch size."""
    n = ctypes.c_int32()
    _check(lib().orca_iteration_wait(eng, ctypes.byref(n), batch_idx, next_tokens), eng)
    return n.value


def orca_last_descriptor(eng, capacity: int):
    nb, nr = ctypes.c_int32(), ctypes.c_int32()
    row_off = (ctypes.c_int32 * (capacity + 1))()
    row_pos = (ctypes.c_int32 * (capacity + 1))()
    row_slot = (ctypes.c_int32 * (capacity + 1))()
    last_row = (ctypes.c_int32 * (capacity + 1))()
    _check(lib().orca_last_descriptor(eng, ctypes.byref(nb), ctypes.byref(nr), row_off, row_pos, row_slot,
                                      last_row, capacity + 1), eng)
    B, N = nb.value, nr.value
    return {"n_batch": B, "n_rows": N, "row_off": list(row_off[:B + 1]), "row_pos": list(row_pos[:N]),
            "row_slot": list(row_slot[:N]), "last_row": list(last_row[:B])}


def orca_last_transfer(eng):
    """(h2d_bytes, d2h_bytes, n_work) of the last orca_iteration."""
    a, b, n = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    _check(lib().orca_last_transfer(eng, ctypes.byref(a), ctypes.byref(b), ctypes.byref(n)), eng)
    return a.value, b.value, n.value


def orca_last_launches(eng) -> int:
    n = ctypes.c_int32()
    _check(lib().orca_last_launches(eng, ctypes.byref(n)), eng)
    return n.value


def orca_attention_workspace_bytes(n_batch: int, n_rows: int, n_heads: int, head_dim: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().orca_attention_workspace_bytes(n_batch, n_rows, n_heads, head_dim, ctypes.byref(n)))
    return n.value


def _i32_arr(vals):
    return (ctypes.c_int32 * len(vals))(*[int(v) for v in vals])


def _i64_arr(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def orca_attention(dtype: int, n_heads: int, head_dim: int, n_slots: int, q_ptr: int, k_ptr: int, v_ptr: int,
                   out_ptr: int, row_off, ctx, slot_base, ws_ptr: int, ws_bytes: int, status_ptr: int,
                   stream=0) -> None:
    nb = len(ctx)
    _check(lib().orca_attention(dtype, n_heads, head_dim, n_slots, ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr),
                                ctypes.c_void_p(v_ptr), ctypes.c_void_p(out_ptr), nb, _i32_arr(row_off),
                                _i32_arr(ctx), _i64_arr(slot_base), ctypes.c_void_p(ws_ptr), ws_bytes,
                                ctypes.c_void_p(status_ptr), ctypes.c_void_p(stream or None)))


def orca_attention_noalloc(dtype: int, n_heads: int, head_dim: int, n_slots: int, q_ptr: int, k_ptr: int,
                           v_ptr: int, out_ptr: int, row_off, ctx, slot_base, status_ptr: int, stream=0) -> None:
    """orca_attention with the library's fixed 8 MiB device scratch, for
    callers that cannot allocate device memory; ORCA_EBATCH if the batch
    needs more scratch than that."""
    nb = len(ctx)
    _check(lib().orca_attention_noalloc(dtype, n_heads, head_dim, n_slots, ctypes.c_void_p(q_ptr),
                                        ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr), ctypes.c_void_p(out_ptr), nb,
                                        _i32_arr(row_off), _i32_arr(ctx), _i64_arr(slot_base),
                                        ctypes.c_void_p(status_ptr), ctypes.c_void_p(stream or None)))


def orca_argmax_rows(logits_ptr: int, n_rows: int, vocab: int, out_ptr: int, stream=0) -> None:
    _check(lib().orca_argmax_rows(ctypes.c_void_p(logits_ptr), n_rows, vocab, ctypes.c_void_p(out_ptr),
                                  ctypes.c_void_p(stream or None)))


def orca_selftest_wait_timeout(status_ptr: int, stream=0) -> None:
    """Enqueue one CTA whose bounded wait expires (about 2 s): it ORs 1
    into the device status word and ends."""
    _check(lib().orca_selftest_wait_timeout(ctypes.c_void_p(status_ptr), ctypes.c_void_p(stream or None)))


ORCA_LINEAR_STORE, ORCA_LINEAR_GELU, ORCA_LINEAR_RESID, ORCA_LINEAR_F32OUT = 0, 1, 2, 3


def orca_linear(dtype: int, mode: int, a_ptr: int, w_ptr: int, bias_ptr: int, out_ptr: int, M: int, N: int, K: int,
                status_ptr: int, stream=0, scratch_ptr: int = 0, scratch_bytes: int = 0, argmax_ptr: int = 0) -> None:
    _check(lib().orca_linear(dtype, mode, ctypes.c_void_p(a_ptr), ctypes.c_void_p(w_ptr),
                             ctypes.c_void_p(bias_ptr or None), ctypes.c_void_p(out_ptr or None), M, N, K,
                             ctypes.c_void_p(scratch_ptr or None), scratch_bytes, ctypes.c_void_p(argmax_ptr or None),
                             ctypes.c_void_p(status_ptr), ctypes.c_void_p(stream or None)))


def argmax_key_column(key: int) -> int:
    """Column of a packed greedy-choice key (see orca_linear), -1 for none."""
    key = int(key) & 0xFFFFFFFFFFFFFFFF
    return -1 if key == 0 else 0xFFFFFFFF - (key & 0xFFFFFFFF)


def orca_gemm_plan_query(M: int, N: int, K: int, n_sms: int, with_scratch: bool = True) -> dict:
    """How the library plans a bf16 M x N x K Linear on a GPU of n_sms SMs
    (host only; see orca.h)."""
    r = orca_gemm_plan_info()
    _check(lib().orca_gemm_plan_query(M, N, K, n_sms, int(bool(with_scratch)), ctypes.byref(r)))
    return {k: getattr(r, k) for k, _ in orca_gemm_plan_info._fields_}


def orca_gemm_pair_segments(M: int, N: int, K: int, n_pairs: int, with_split: bool, pair: int) -> list:
    """The CTA-pair GEMM's work for one pair, in order: rows of (tile, row tile,
    column tile, k-block begin, end, pairs sharing the tile, place in k order,
    counter pair or -1, partial slot or -1) (host only; see orca.h)."""
    n = lib().orca_gemm_pair_segments(M, N, K, n_pairs, int(bool(with_split)), pair, None, 0)
    if n < 0:
        _check(n)
    buf = (ctypes.c_int32 * (9 * max(1, n)))()
    m = lib().orca_gemm_pair_segments(M, N, K, n_pairs, int(bool(with_split)), pair, buf, n)
    if m != n:
        raise OrcaError(ORCA_EINVAL, f"orca_gemm_pair_segments: {m} segments, expected {n}")
    return [tuple(buf[9 * i:9 * i + 9]) for i in range(n)]


def orca_profile_enable(eng, mode: int) -> None:
    """mode 0 off, 1 CUDA events around eager launches, 2 launch stamps in
    the graph-replayed forward (True / False mean 1 / 0)."""
    _check(lib().orca_profile_enable(eng, int(mode)), eng)


def orca_profile_read(eng, kernel_class: int) -> dict:
    s = orca_kernel_stats()
    _check(lib().orca_profile_read(eng, kernel_class, ctypes.byref(s)), eng)
    return {"launches": s.launches, "total_ms": s.total_ms, "flops": s.flops, "bytes": s.bytes}


def orca_last_error(eng) -> str:
    buf = ctypes.create_string_buffer(512)
    lib().orca_last_error(eng, buf, 512)
    return buf.value.decode(errors="replace")

"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This module holds no arithmetic of the method itself: it only draws random
weights, request traces and token streams from numpy's PCG64 generator, so
that the CPU oracle and the CUDA path see exactly the same inputs.  Nothing
here computes a layer, an attention score or a scheduling decision.

Model shapes follow the GPT family the Orca evaluation uses ("Orca: iteration-
level scheduling", environment section: GPT-3-family models); the request
trace follows the same page's synthetic workload (input lengths uniform,
output lengths uniform, Poisson arrivals, no end-of-sequence token).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

DTYPE_F32 = 0
DTYPE_BF16 = 1


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_heads: int
    ffn: int
    vocab: int
    max_pos: int
    dtype: int  # DTYPE_F32 or DTYPE_BF16

    @property
    def head_dim(self) -> int:
        return self.hidden // self.n_heads


# Toy GPT: 2 layers, H=64, 4 heads, vocab 256, fp32.
TOY = ModelShape(n_layers=2, hidden=64, n_heads=4, ffn=256, vocab=256, max_pos=64, dtype=DTYPE_F32)
# GPT-2-small-shaped decoder in bf16.
GPT2_SMALL = ModelShape(n_layers=12, hidden=768, n_heads=12, ffn=3072, vocab=50257, max_pos=1024,
                        dtype=DTYPE_BF16)
# 13B-shaped decoder in bf16 (40 layers, H=5120, 40 heads, FFN 4H).
GPT_13B = ModelShape(n_layers=40, hidden=5120, n_heads=40, ffn=20480, vocab=50257, max_pos=4352,
                     dtype=DTYPE_BF16)


def with_layers(shape: ModelShape, n_layers: int) -> ModelShape:
    return dataclasses.replace(shape, n_layers=n_layers)


def with_dtype(shape: ModelShape, dtype: int) -> ModelShape:
    return dataclasses.replace(shape, dtype=dtype)


LAYER_TENSORS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                 "ln2_g", "ln2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2")
GLOBAL_TENSORS = ("tok_emb", "pos_emb", "lnf_g", "lnf_b")


def layer_tensor_shapes(s: ModelShape) -> Dict[str, tuple]:
    """Per-layer tensors.  Matrices are stored [out_features, in_features]."""
    H, F = s.hidden, s.ffn
    return {
        "ln1_g": (H,), "ln1_b": (H,),
        "w_qkv": (3 * H, H), "b_qkv": (3 * H,),
        "w_o": (H, H), "b_o": (H,),
        "ln2_g": (H,), "ln2_b": (H,),
        "w_fc1": (F, H), "b_fc1": (F,),
        "w_fc2": (H, F), "b_fc2": (H,),
    }


def global_tensor_shapes(s: ModelShape) -> Dict[str, tuple]:
    return {"tok_emb": (s.vocab, s.hidden), "pos_emb": (s.max_pos, s.hidden),
            "lnf_g": (s.hidden,), "lnf_b": (s.hidden,)}


def is_matrix(name: str) -> bool:
    """Matrices and embedding tables are stored in the model dtype; LayerNorm
    parameters and biases are always stored in fp32."""
    return name.startswith("w_") or name.endswith("_emb")


def to_storage(a: np.ndarray, dtype: int) -> np.ndarray:
    """Return fp32 values exactly representable in the storage dtype.

    bf16 storage rounds with torch's round-to-nearest-even conversion; the
    returned array is still float32 (the bf16 values widened exactly)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype == DTYPE_F32:
        return a
    import torch
    return torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of fp32 values that are exactly bf16."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values are not exactly representable in bf16")
    return (u >> 16).astype(np.uint16)


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def make_weights(shape: ModelShape, seed: int = 0, w_std: float = 0.02, bias_std: float = 0.0,
                 ln_std: float = 0.0, layers: Optional[List[int]] = None) -> Dict[str, np.ndarray]:
    """Random-init GPT weights as fp32 arrays holding storage-dtype values.

    Matrices and embeddings ~ N(0, w_std^2); biases ~ N(0, bias_std^2);
    LayerNorm gamma = 1 + N(0, ln_std^2), beta ~ N(0, ln_std^2).  With the
    default bias_std = ln_std = 0 this is the plain GPT initialisation
    (biases 0, gamma 1, beta 0).  Each tensor has its own PCG64 stream keyed
    by (seed, layer, tensor index), so a slice of layers is reproducible
    without generating the others.  Keys: "tok_emb", ..., "L{l}.w_qkv", ...
    """
    out: Dict[str, np.ndarray] = {}
    gshapes = global_tensor_shapes(shape)
    for ti, name in enumerate(GLOBAL_TENSORS):
        out[name] = _draw(name, gshapes[name], _rng(seed, 1_000_000, ti), shape.dtype,
                          w_std, bias_std, ln_std)
    lshapes = layer_tensor_shapes(shape)
    for l in (range(shape.n_layers) if layers is None else layers):
        for ti, name in enumerate(LAYER_TENSORS):
            out[f"L{l}.{name}"] = _draw(name, lshapes[name], _rng(seed, l, ti), shape.dtype,
                                        w_std, bias_std, ln_std)
    return out


def _draw(name, shp, rng, dtype, w_std, bias_std, ln_std) -> np.ndarray:
    z = rng.standard_normal(shp, dtype=np.float32)
    if is_matrix(name):
        return to_storage(z * np.float32(w_std), dtype)
    if name.endswith("_g"):
        return (np.float32(1.0) + z * np.float32(ln_std)).astype(np.float32)
    if name.endswith("_b") and name.startswith("ln"):
        return (z * np.float32(ln_std)).astype(np.float32)
    return (z * np.float32(bias_std)).astype(np.float32)  # linear biases


@dataclasses.dataclass
class Request:
    req_id: int
    arrival: int            # arrival iteration index (or any monotone clock)
    prompt: np.ndarray      # int32 token ids
    out_len: int            # tokens to generate (no end-of-sequence token)
    max_tokens: int         # K/V slots reserved on first schedule
    forced: Optional[np.ndarray] = None  # int32 continuation for teacher forcing

    @property
    def n_prompt(self) -> int:
        return int(self.prompt.shape[0])


def poisson_arrivals(n: int, rate_per_iter: float, rng: np.random.Generator) -> np.ndarray:
    """Arrival iteration indices of a Poisson process (exponential gaps),
    floored to integers; rate_per_iter = inf puts every request at 0."""
    if not np.isfinite(rate_per_iter):
        return np.zeros(n, dtype=np.int64)
    gaps = rng.exponential(1.0 / rate_per_iter, size=n)
    return np.floor(np.cumsum(gaps) - gaps[0]).astype(np.int64)


def make_trace(n_requests: int, prompt_range, out_range, vocab: int, seed: int = 0,
               rate_per_iter: float = float("inf"), max_extra: Optional[int] = None,
               forced: bool = False) -> List[Request]:
    """Synthetic request trace.

    prompt_range / out_range are inclusive (lo, hi) for uniform integer draws;
    token ids are uniform in [0, vocab).  max_tokens = prompt + max_extra when
    max_extra is given, else prompt + out_len.  forced=True also draws an
    out_len-long uniform continuation used as the teacher-forced stream."""
    rng = _rng(seed, 2_000_000)
    arr = poisson_arrivals(n_requests, rate_per_iter, rng)
    reqs = []
    for i in range(n_requests):
        lp = int(rng.integers(prompt_range[0], prompt_range[1] + 1))
        lo = int(rng.integers(out_range[0], out_range[1] + 1))
        prompt = rng.integers(0, vocab, size=lp, dtype=np.int64).astype(np.int32)
        cont = rng.integers(0, vocab, size=lo, dtype=np.int64).astype(np.int32) if forced else None
        mt = lp + (max_extra if max_extra is not None else lo)
        reqs.append(Request(req_id=i, arrival=int(arr[i]), prompt=prompt, out_len=lo,
                            max_tokens=mt, forced=cont))
    return reqs


def figure5_trace(vocab: int = 256, seed: int = 0, out_len: int = 8, extra: int = 10) -> List[Request]:
    """The four requests of the Orca Figure 5 batch.

    x1 (3-token prompt) and x2 (1-token prompt) arrive at iteration 0 and are
    prefilled there; x3 (2-token prompt) and x4 (3-token prompt) arrive at
    iteration 1.  Iteration 1 is then the Figure 5 batch: x1 decodes with 3
    cached tokens, x2 with 1 cached, x3 prefills 2 tokens, x4 prefills 3."""
    rng = _rng(seed, 3_000_000)
    spec = [(0, 3), (0, 1), (1, 2), (1, 3)]
    reqs = []
    for i, (arrival, lp) in enumerate(spec):
        prompt = rng.integers(0, vocab, size=lp, dtype=np.int64).astype(np.int32)
        reqs.append(Request(req_id=i, arrival=arrival, prompt=prompt, out_len=out_len,
                            max_tokens=lp + extra))
    return reqs


def mixed_batch_lengths(n_prefill: int, prompt_range, n_decode: int, ctx_range, seed: int = 0):
    """Lengths of one fixed mixed iteration: n_prefill prompt lengths and
    n_decode cached-context lengths, each uniform over its inclusive range."""
    rng = _rng(seed, 5_000_000)
    prompts = rng.integers(prompt_range[0], prompt_range[1] + 1, size=n_prefill).astype(np.int64)
    ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=n_decode).astype(np.int64)
    return prompts, ctx


def token_ids(n: int, vocab: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """n token ids uniform in [0, vocab) (int32)."""
    return _rng(seed, 6_000_000, stream).integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def random_kv(n_tokens: int, hidden: int, seed: int, dtype: int) -> np.ndarray:
    """[n_tokens, hidden] random values (N(0,1)) in storage precision, used to
    fill K/V slots directly when an attention case needs long cached contexts."""
    z = _rng(seed, 4_000_000).standard_normal((n_tokens, hidden), dtype=np.float32)
    return to_storage(z, dtype)

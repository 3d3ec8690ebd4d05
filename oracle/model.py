"""Per-request, token-at-a-time GPT generation: what selective batching must match.

The block follows the GPT family of the Orca evaluation (Orca walk-through,
"环境与模型配置"): learned token and position embeddings, pre-LayerNorm blocks
with a QKV Linear, attention, an attention-out Linear, residual Adds, an MLP
of two Linears around GeLU, a final LayerNorm and an LM head tied to the
token embedding.  Attention of a token reads the K/V of its own request's
earlier tokens and of itself (Figure 5: x1 attends over x11, x12, x13 and the
current token).  Greedy decoding takes the lowest index among equal maxima
(CS349D Lecture 2, section 4.2: the greedily chosen next tokens match).

Weights are stored [out_features, in_features]; y = W x + b.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from .numerics import gelu_tanh, layer_norm, round_bf16, softmax

_BF16 = 1


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_heads: int) -> np.ndarray:
    """Multi-head attention of one query row over keys K[0..T), values V[0..T).

    Per head h: softmax(q_h . K_h^T / sqrt(d)) . V_h; heads concatenated
    (Figure 5: one request's query against its own cached K/V)."""
    H = q.shape[-1]
    d = H // n_heads
    out = np.empty(H)
    scale = 1.0 / np.sqrt(d)
    for h in range(n_heads):
        sl = slice(h * d, (h + 1) * d)
        p = softmax(K[:, sl] @ q[sl] * scale)
        out[sl] = p @ V[:, sl]
    return out


class GPTOracle:
    def __init__(self, shape, weights: Dict[str, np.ndarray], layers: Optional[Sequence[int]] = None):
        self.shape = shape
        self.H = shape.hidden
        self.nh = shape.n_heads
        self.d = shape.hidden // shape.n_heads
        self.bf16 = shape.dtype == _BF16
        self.layers = list(range(shape.n_layers) if layers is None else layers)
        f64 = lambda a: np.asarray(a, dtype=np.float64)
        self.tok_emb = f64(weights["tok_emb"])
        self.pos_emb = f64(weights["pos_emb"])
        self.lnf_g = f64(weights["lnf_g"])
        self.lnf_b = f64(weights["lnf_b"])
        self.L = []
        for l in self.layers:
            self.L.append({k: f64(weights[f"L{l}.{k}"]) for k in
                           ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                            "ln2_g", "ln2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2")})

    # bf16 rounding at the points where the CUDA path stores bf16
    def _r(self, x: np.ndarray) -> np.ndarray:
        return round_bf16(x) if self.bf16 else x

    def new_cache(self, capacity: int) -> dict:
        """Per-request K/V cache: one [capacity, H] K and V array per layer."""
        return {"n": 0,
                "k": [np.zeros((capacity, self.H)) for _ in self.layers],
                "v": [np.zeros((capacity, self.H)) for _ in self.layers]}

    def attend(self, q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
        return attend(q, K, V, self.nh)

    def step(self, cache: dict, token: int, pos: int, want_logits: bool = True) -> Optional[np.ndarray]:
        """Feed one token at position `pos`; append its K/V to the cache;
        return the next-token logits (float64 [vocab]) if asked."""
        assert pos == cache["n"], "tokens of a request are fed in order"
        H = self.H
        x = self.tok_emb[token] + self.pos_emb[pos]
        for li, w in enumerate(self.L):
            h = self._r(layer_norm(x, w["ln1_g"], w["ln1_b"]))
            qkv = w["w_qkv"] @ h + w["b_qkv"]
            q = self._r(qkv[:H])
            cache["k"][li][pos] = self._r(qkv[H:2 * H])
            cache["v"][li][pos] = self._r(qkv[2 * H:])
            a = self._r(self.attend(q, cache["k"][li][:pos + 1], cache["v"][li][:pos + 1]))
            x = x + (w["w_o"] @ a + w["b_o"])
            h2 = self._r(layer_norm(x, w["ln2_g"], w["ln2_b"]))
            u = self._r(gelu_tanh(w["w_fc1"] @ h2 + w["b_fc1"]))
            x = x + (w["w_fc2"] @ u + w["b_fc2"])
        cache["n"] = pos + 1
        if not want_logits:
            return None
        hf = self._r(layer_norm(x, self.lnf_g, self.lnf_b))
        return self.tok_emb @ hf

    def generate(self, prompt: Sequence[int], out_len: int, forced: Optional[Sequence[int]] = None,
                 keep_logits: bool = True, stop_after: Optional[int] = None):
        """Generate `out_len` tokens for one request, alone.

        The prompt is fed one token at a time; its last token yields the first
        generated token.  Each later step feeds the previous token: the
        previous greedy token, or forced[k-1] under teacher forcing.
        Returns (greedy tokens [out_len], logits list or None, fed tokens).
        `stop_after` ends early after that many generated tokens."""
        n_gen = out_len if stop_after is None else min(out_len, stop_after)
        cache = self.new_cache(len(prompt) + out_len)
        logits: List[np.ndarray] = []
        greedy: List[int] = []
        fed: List[int] = []
        lg = None
        for t, tok in enumerate(prompt):
            lg = self.step(cache, int(tok), t, want_logits=(t == len(prompt) - 1))
        for k in range(n_gen):
            if k > 0:
                tok = int(forced[k - 1]) if forced is not None else greedy[-1]
                fed.append(tok)
                lg = self.step(cache, tok, len(prompt) + k - 1)
            greedy.append(int(np.argmax(lg)))
            if keep_logits:
                logits.append(lg)
        return greedy, (logits if keep_logits else None), fed


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Row-wise argmax, lowest index among equal maxima."""
    return np.argmax(logits, axis=-1)

"""Elementwise numerics of the oracle, float64 throughout.

The GPT block names LayerNorm, GeLU, Linear and Add as its token-wise
operators (Orca walk-through, "观察：并非所有算子都要求"请求边界"").  The pages do
not fix epsilon or the GeLU form; the GPT convention is used: epsilon 1e-5
with the biased variance, and the tanh approximation of GeLU.
"""
import numpy as np

LN_EPS = 1e-5


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits.  With x = m * 2**e, 0.5 <= |m| < 1
    (frexp), the kept value is rint(m * 2**8) / 2**8 * 2**e, and rint rounds
    half to even.  Values that overflow bf16 or fall in its subnormal range
    do not occur in these models and are not special-cased."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray) -> np.ndarray:
    """(x - mean) / sqrt(var + eps) * gamma + beta over the last axis,
    biased variance."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + LN_EPS) * gamma + beta


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def softmax(s: np.ndarray) -> np.ndarray:
    """Softmax over the last axis (shifted by the max for range only)."""
    z = np.exp(s - s.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)

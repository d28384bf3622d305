"""Elementary operations of the draft layer, in float64.

[NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
section "Eagle3 Draft Model Architecture": RMSNorm (input_layernorm,
hidden_norm, post_attention_layernorm, final norm), shared rotary embeddings,
and the Llama MLP.  The pages name these operations without formulas; the
forms used here are the standard Llama ones (stated readings):

* RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g
* rotary embedding: rotate-half pairing (i, i + d/2), angle pos * theta^(-2i/d)
* MLP: down(silu(gate(x)) * up(x))
"""
import numpy as np


def to_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits.  ``frexp`` gives x = m * 2**e with
    0.5 <= |m| < 1, so the significand to keep is m * 2**8 rounded to an
    integer; ``rint`` rounds halves to even.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def rmsnorm(x, g, eps):
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def rope(x, pos, theta):
    """Rotary embedding on the last axis of ``x`` ``[..., d]`` at integer positions ``pos``.

    ``pos`` broadcasts against ``x.shape[:-1]``.  Pairs (i, i + d/2) rotate by
    angle pos * theta**(-2i/d).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def logsumexp(x, axis=-1):
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=axis, keepdims=True)
    return (m + np.log(np.sum(np.exp(x - m), axis=axis, keepdims=True))).squeeze(axis)


def topk_desc(values, k):
    """Indices of the k largest entries of each row; larger value first, equal values
    in ascending index order (the stated tie-break)."""
    v = np.asarray(values)
    idx = np.arange(v.shape[-1])
    out = np.empty(v.shape[:-1] + (k,), dtype=np.int64)
    flat_v = v.reshape(-1, v.shape[-1])
    flat_o = out.reshape(-1, k)
    for r in range(flat_v.shape[0]):
        order = np.lexsort((idx, -flat_v[r]))
        flat_o[r] = order[:k]
    return out

"""A second, independent formulation of the decode step, used to pin the oracle.

This is the full-sequence causal form of the LLaMA forward pass as the page
"LLaMA implemented in R Tensorflow and Keras" writes it (TransformerDecoder
``call``): every position is recomputed from scratch with batched matrix
products, a -Inf upper-triangle mask (``make_mask``), RoPE applied in tensor
form (``precompute_rotarty_freqs`` + ``apply_rotary_embedding`` with
``rotate_every_two``), and softmax over the masked score matrix.  It keeps
everything in float64 and never touches a KV cache, so incremental decoding
in the oracle must reproduce its logits at every position.

Two deliberate differences from that page, both matching the llama2.c pages
that the oracle follows: RMSNorm eps is 1e-5, and K/V heads are shared by
query heads through the map g(h) = floor(h * n_kv_heads / n_heads) (the
R page has no grouped-query attention).
"""
from __future__ import annotations

import numpy as np


def rotary_tables(seqlen: int, head_size: int, theta: float = 10000.0):
    """cos/sin tables (seqlen, head_size), each pair's angle repeated twice."""
    t = np.arange(seqlen, dtype=np.float64)
    freqs = np.arange(0.0, 1.0, 1.0 / (head_size // 2), dtype=np.float64)[: head_size // 2]
    freqs = 1.0 / (theta ** freqs)
    ang = np.einsum("a,b->ab", t, freqs)
    return np.repeat(np.cos(ang), 2, axis=-1), np.repeat(np.sin(ang), 2, axis=-1)


def rotate_every_two(x: np.ndarray) -> np.ndarray:
    x1 = x[..., 0::2]
    x2 = x[..., 1::2]
    return np.stack([-x2, x1], axis=-1).reshape(x.shape)


def apply_rotary(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """x (T, heads, hs); cos/sin (T, hs)."""
    return x * cos[:, None, :] + rotate_every_two(x) * sin[:, None, :]


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w


def causal_mask(seqlen: int) -> np.ndarray:
    i = np.arange(seqlen)[:, None]
    j = np.arange(seqlen)[None, :]
    return np.where(i < j, -np.inf, 0.0)


def softmax_last(s: np.ndarray) -> np.ndarray:
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def full_logits(config: tuple, weights: dict, tokens, return_probs: bool = False):
    """Logits (T, vocab) for every prefix of ``tokens``; optionally the
    attention probabilities (layer, head, T, T)."""
    dim, hidden, L, H, KV, V, S = config
    hs = dim // H
    W = {k: np.asarray(v, dtype=np.float64) for k, v in weights.items()}
    toks = np.asarray(tokens)
    T = toks.size
    cos, sin = rotary_tables(T, hs)
    mask = causal_mask(T)
    group = (np.arange(H) * KV) // H
    x = W["emb"][toks]
    probs = []
    for l in range(L):
        h = rms_norm(x, W["rms_att"][l])
        q = (h @ W["wq"][l].T).reshape(T, H, hs)
        k = (h @ W["wk"][l].T).reshape(T, KV, hs)
        v = (h @ W["wv"][l].T).reshape(T, KV, hs)
        q = apply_rotary(q, cos, sin)
        k = apply_rotary(k, cos, sin)
        k = k[:, group, :]
        v = v[:, group, :]
        scores = np.einsum("thd,shd->hts", q, k) / np.sqrt(hs) + mask
        p = softmax_last(scores)
        probs.append(p)
        o = np.einsum("hts,shd->thd", p, v).reshape(T, dim)
        x = x + o @ W["wo"][l].T
        h = rms_norm(x, W["rms_ffn"][l])
        a = h @ W["w1"][l].T
        b = h @ W["w3"][l].T
        x = x + ((a / (1.0 + np.exp(-a))) * b) @ W["w2"][l].T
    x = rms_norm(x, W["rms_final"])
    logits = x @ W["wcls"].T
    return (logits, np.stack(probs)) if return_probs else logits

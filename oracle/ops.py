"""The decode step's per-token operations, plain fp64.

Pages: the pure C + CUDA inference engine page, section 4.4 (custom CUDA
operators) names every op here: single-token GEMV, fused RMSNorm, RoPE with a
precomputed sin/cos table, SwiGLU fused with the projection, and a causal
softmax with the mask applied inside it; section 1 names GQA and the KV cache.
The pages give no formulas, so each function states the standard Llama
definition it writes out and the reading taken where the pages are silent.
"""
from __future__ import annotations

import numpy as np


def round_f16(x: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16 (nearest, ties to even) and back to fp64.

    The KV cache is fp16, so the oracle stores exactly what the cache holds.
    """
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * g, over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def rope_angles(pos, head_dim: int, theta: float) -> np.ndarray:
    """Angle of pair i at position pos: pos * theta^(-2i/head_dim), i < head_dim/2."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return np.multiply.outer(np.asarray(pos, dtype=np.float64), inv_freq)


def rope(v: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate each adjacent pair (2i, 2i+1) of every head vector by pos*theta_i.

    v: [..., n_heads, head_dim] for one position, or [T, n_heads, head_dim]
    with pos an array of T positions.  Reading (the pages are silent on the
    pairing): adjacent pairs, the layout of GGUF Llama models the engine page
    loads; (a, b) -> (a cos - b sin, a sin + b cos).
    """
    v = np.asarray(v, dtype=np.float64)
    hd = v.shape[-1]
    ang = rope_angles(pos, hd, theta)          # [hd/2] or [T, hd/2]
    if ang.ndim == 2:
        ang = ang[:, None, :]                  # broadcast over heads
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., 0::2], v[..., 1::2]
    out = np.empty_like(v)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def softmax(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """GQA attention of one query position over its cached keys.

    q: [n_heads, hd]; k, v: [n, n_kv_heads, hd] holding positions 0..n-1 (the
    causal range: the new token's own key is already appended).  Readings:
    query head h reads KV head floor(h / (n_heads / n_kv_heads)); scores are
    scaled by 1/sqrt(hd).  Returns o: [n_heads, hd].
    """
    nh, hd = q.shape
    nkv = k.shape[1]
    g = nh // nkv
    o = np.empty((nh, hd), dtype=np.float64)
    for h in range(nh):
        kv = h // g
        s = k[:, kv, :] @ q[h] / np.sqrt(hd)
        o[h] = softmax(s) @ v[:, kv, :]
    return o


def attention_partial(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """The softmax statistics of one query position over a subset of its keys
    (the form in which attention over a shared prefix and over each branch's
    own positions are computed apart and then merged: cascade attention for
    the branches of a fork, which read one prefix).

    q: [n_heads, hd]; k, v: [n, n_kv_heads, hd] (n may be 0).  Returns
    (o, m, l): per head the running maximum m of the scaled scores, the sum
    l of exp(score - m) and the unnormalised o = sum exp(score - m) v; an
    empty key set gives m = -inf, l = 0, o = 0.
    """
    nh, hd = q.shape
    nkv = k.shape[1]
    g = nh // nkv
    o = np.zeros((nh, hd), dtype=np.float64)
    m = np.full(nh, -np.inf)
    l = np.zeros(nh)
    if k.shape[0] == 0:
        return o, m, l
    for h in range(nh):
        kv = h // g
        s = k[:, kv, :] @ q[h] / np.sqrt(hd)
        m[h] = np.max(s)
        e = np.exp(s - m[h])
        l[h] = np.sum(e)
        o[h] = e @ v[:, kv, :]
    return o, m, l


def merge_partials(parts) -> np.ndarray:
    """Attention output from the statistics of disjoint key subsets that
    together cover the key range: rescale every part to the common maximum
    and divide the summed outputs by the summed weights."""
    ms = np.stack([p[1] for p in parts])                 # [parts, n_heads]
    mx = np.max(ms, axis=0)
    scale = np.where(np.isfinite(ms), np.exp(ms - mx[None, :]), 0.0)
    o = sum(sc[:, None] * p[0] for sc, p in zip(scale, parts))
    l = sum(sc * p[2] for sc, p in zip(scale, parts))
    return o / l[:, None]


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos0: int = 0) -> np.ndarray:
    """Attention of T query positions q_pos0 .. q_pos0+T-1 over keys 0..n-1.

    q: [T, n_heads, hd]; k, v: [n, n_kv_heads, hd].  Query t sees keys
    j <= q_pos0 + t (the causal mask applied inside the softmax).
    """
    T, nh, hd = q.shape
    n, nkv, _ = k.shape
    g = nh // nkv
    o = np.empty((T, nh, hd), dtype=np.float64)
    qpos = q_pos0 + np.arange(T)
    mask = np.arange(n)[None, :] > qpos[:, None]          # [T, n] True = hidden
    for h in range(nh):
        kv = h // g
        s = q[:, h, :] @ k[:, kv, :].T / np.sqrt(hd)       # [T, n]
        s = np.where(mask, -np.inf, s)
        o[:, h, :] = softmax(s) @ v[:, kv, :]
    return o


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """h = silu(gate) * up."""
    return silu(gate) * np.asarray(up, dtype=np.float64)


def greedy(logits: np.ndarray) -> int:
    """argmax; ties go to the lowest index."""
    return int(np.argmax(np.asarray(logits)))


def top2_gap(logits: np.ndarray) -> float:
    """Difference between the largest and second-largest logit."""
    part = np.partition(np.asarray(logits, dtype=np.float64), -2)
    return float(part[-1] - part[-2])


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    """Cosine similarity a.b / (|a| |b|) of two vectors (0 if either is zero)."""
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.sqrt(a @ a), np.sqrt(b @ b)
    return float(a @ b / (na * nb)) if na > 0 and nb > 0 else 0.0

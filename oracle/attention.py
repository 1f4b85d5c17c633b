"""Decode attention in fp64: the plain definition and the forms it must agree with.

Definition ("企业官网建设流程全解析" (KV Cache 原理篇) §1.2):
``Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V``.  In decode one new
query token per sequence attends over every cached token of its own
sequence, including the token appended this step (§3.2 of the same page:
K and V are appended first, then Q attends over history plus the current
token), so no mask is needed.  The scale is passed in (the fp32 value of
``1/sqrt(d)`` by default).

GQA ("企业官网建设流程全解析" §2.2, "KV Cache优化实战" §2.1): several query
heads share one KV head; with ``G = Hq / Hkv`` the reading adopted is the
contiguous grouping, query head ``h`` uses KV head ``h // G``.

Numerical stabilisation subtracts the row maximum, as the NumPy
demonstration of "企业官网建设流程全解析" §5.2 does; in fp64 this changes
nothing beyond rounding.
"""
from __future__ import annotations

import math

import numpy as np


def decode_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Attention of one sequence's new query over its cached tokens.

    q: [Hq, D]; K, V: [L, Hkv, D] (any float type, used in fp64).
    Returns fp64 [Hq, D]; all zeros when L == 0.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hq, d = q.shape
    length, hkv, _ = K.shape
    if hq % hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = hq // hkv
    out = np.zeros((hq, d))
    if length == 0:
        return out
    for h in range(hq):
        kv = h // group
        s = float(scale) * (K[:, kv, :] @ q[h])
        s = s - s.max()
        p = np.exp(s)
        out[h] = (p @ V[:, kv, :]) / p.sum()
    return out


def decode_attention_loops(q, K, V, scale) -> np.ndarray:
    """The same quantity with explicit Python loops (tiny inputs only)."""
    hq, d = len(q), len(q[0])
    length, hkv = len(K), len(K[0]) if len(K) else 1
    group = hq // hkv
    out = [[0.0] * d for _ in range(hq)]
    if length == 0:
        return np.array(out)
    for h in range(hq):
        kv = h // group
        scores = []
        for j in range(length):
            acc = 0.0
            for c in range(d):
                acc += float(q[h][c]) * float(K[j][kv][c])
            scores.append(float(scale) * acc)
        mx = max(scores)
        w = [math.exp(s - mx) for s in scores]
        tot = sum(w)
        for c in range(d):
            acc = 0.0
            for j in range(length):
                acc += w[j] * float(V[j][kv][c])
            out[h][c] = acc / tot
    return np.array(out)


def causal_attention_all_positions(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Full recompute without a cache: every position attends to itself and the past.

    Q: [T, Hq, D]; K, V: [T, Hkv, D].  Returns [T, Hq, D].  This is the
    no-cache path of "KV Cache 与 vLLM" (zwxr.cn) §1.2 / §1.3 (the whole
    sequence re-run with a causal mask); row t must equal the decode of
    position t over a cache holding tokens 0..t.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    t_len, hq, d = Q.shape
    hkv = K.shape[1]
    group = hq // hkv
    mask = np.triu(np.full((t_len, t_len), -np.inf), k=1)
    out = np.empty((t_len, hq, d))
    for h in range(hq):
        kv = h // group
        scores = float(scale) * (Q[:, h, :] @ K[:, kv, :].T) + mask
        scores = scores - scores.max(axis=1, keepdims=True)
        w = np.exp(scores)
        w = w / w.sum(axis=1, keepdims=True)
        out[:, h, :] = w @ V[:, kv, :]
    return out


def split_partials(q, K, V, scale, bounds):
    """Unnormalised partial results over token ranges ``bounds = [(start, stop), ...]``.

    For each range: ``m`` = max score, ``l = sum exp(s - m)``,
    ``o = sum exp(s - m) v`` (per query head).  Empty ranges give
    ``m = -inf, l = 0, o = 0``.  This is the split-KV contract the decode
    path uses for long contexts; it is checked against the unsplit
    definition.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hq, d = q.shape
    hkv = K.shape[1]
    group = hq // hkv
    parts = []
    for start, stop in bounds:
        o = np.zeros((hq, d))
        m = np.full(hq, -np.inf)
        l = np.zeros(hq)
        if stop > start:
            for h in range(hq):
                kv = h // group
                s = float(scale) * (K[start:stop, kv, :] @ q[h])
                m[h] = s.max()
                p = np.exp(s - m[h])
                l[h] = p.sum()
                o[h] = p @ V[start:stop, kv, :]
        parts.append((o, m, l))
    return parts


def lse_merge(parts) -> np.ndarray:
    """Merge partials: ``out = sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s``, M = max_s m_s."""
    o0, m0, _ = parts[0]
    hq, d = o0.shape
    out = np.zeros((hq, d))
    ms = np.stack([p[1] for p in parts])          # [S, Hq]
    big_m = ms.max(axis=0)
    for h in range(hq):
        if not np.isfinite(big_m[h]):
            continue  # every range empty: zero output
        num = np.zeros(d)
        den = 0.0
        for o, m, l in parts:
            if np.isfinite(m[h]):
                w = math.exp(m[h] - big_m[h])
                num += w * o[h]
                den += w * l[h]
        out[h] = num / den
    return out

"""Dense softmax attention in fp64 on the CPU: the plain definition.

TEST INFRASTRUCTURE (see oracle/__init__.py): never imported by the product path.

What the ring computes is, exactly up to rounding order, ordinary softmax
attention over the whole sequence:
  * "Ring Attention" (aarnphm.xyz), ring recurrence display: scores
    S = Q K^T / sqrt(d_h), and O = y / z after every shard was folded in.
  * "Ring Attention: Distributed Attention Across Devices" (aicomputerinstitute),
    "Worked example: tracing the ring by hand": the dense procedure -- subtract
    the row max, exponentiate, divide by the sum, weight V -- and the claim
    that the ring reproduces it.
  * "Ring Attention: what the near-infinite context paper actually says",
    "The ring mechanism, step by step": the result is identical to full-sequence
    attention on one device; "The causal masking complication": query position
    i sees key positions <= i (inclusive diagonal).

Conventions (readings where the pages are silent):
  * Layout: q [B, N, H, d], k and v [B, N, G, d], tokens in original order.
  * Grouped-query attention: query head h reads kv head g = floor(h * G / H).
  * LSE = m + ln z in natural log of the *scaled* scores.
  * A row that admits no key has O = 0 and LSE = -inf (cannot happen under a
    causal mask on the full sequence, since every token sees itself).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


def kv_head_of(h: int, heads: int, kv_heads: int) -> int:
    """Query head h reads kv head floor(h * G / H): consecutive groups of H/G
    query heads share one kv head."""
    return (h * kv_heads) // heads


def default_scale(head_dim: int) -> float:
    """1 / sqrt(d_h) ("Ring Attention" (aarnphm.xyz), definition of S)."""
    return 1.0 / math.sqrt(head_dim)


def attend_rows(q_rows: np.ndarray, K: np.ndarray, V: np.ndarray, allowed: np.ndarray,
                scale: float):
    """Softmax attention of a few query rows over keys K, V with an explicit
    boolean mask `allowed` [rows, keys].

    Returns (O [rows, d], LSE [rows]) in fp64.
    """
    S = (q_rows @ K.T) * scale                       # scaled scores
    S = np.where(allowed, S, -np.inf)
    m = S.max(axis=1)                                # row max over admitted keys
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.exp(S - m_safe[:, None])                  # exp(-inf) = 0 on masked keys
    z = E.sum(axis=1)
    y = E @ V
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(empty[:, None], 0.0, y / np.where(empty, 1.0, z)[:, None])
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, z)))
    return O, lse


def dense_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                    scale: Optional[float] = None, rows: Optional[Sequence[int]] = None,
                    heads: Optional[Sequence[int]] = None, max_chunk_elems: int = 1 << 23):
    """O and LSE of plain softmax attention.

    q [B,N,H,d], k/v [B,N,G,d]: arrays holding the exact input values (any float
    dtype; every slice is converted to fp64 before use).
    rows: optional subset of query tokens (original order) to compute.
    heads: optional subset of query heads to compute.
    Returns O [B, R, Hs, d] and LSE [B, Hs, R] (R = len(rows) or N,
    Hs = len(heads) or H).
    """
    B, N, H, d = q.shape
    rows_ = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    heads_ = list(range(H)) if heads is None else list(heads)
    q_rows = np.asarray(q)[:, rows_][:, :, heads_]
    return attention_at(q_rows, rows_, heads_, H, k, v, causal, scale, max_chunk_elems)


def attention_at(q_rows: np.ndarray, rows: Sequence[int], heads: Sequence[int], n_heads: int,
                 k: np.ndarray, v: np.ndarray, causal: bool, scale: Optional[float] = None,
                 max_chunk_elems: int = 1 << 23):
    """Attention of given query vectors q_rows [B, R, Hs, d], which sit at token
    positions `rows` and belong to query heads `heads` (of n_heads), over all N
    keys of k/v [B, N, G, d]. Returns O [B, R, Hs, d] and LSE [B, Hs, R] in fp64."""
    B, R, Hs, d = q_rows.shape
    N, G = k.shape[1], k.shape[2]
    assert k.shape == (B, N, G, d) and v.shape == (B, N, G, d)
    assert n_heads % G == 0
    if scale is None:
        scale = default_scale(d)
    rows = np.asarray(rows, dtype=np.int64)
    O = np.zeros((B, R, Hs, d))
    LSE = np.zeros((B, Hs, R))
    chunk = max(1, max_chunk_elems // max(N, 1))
    keys = np.arange(N)
    for b in range(B):
        by_g = {}
        for hi, h in enumerate(heads):
            by_g.setdefault(kv_head_of(h, n_heads, G), []).append(hi)
        for g, his in by_g.items():
            K = np.asarray(k[b, :, g, :], dtype=np.float64)
            V = np.asarray(v[b, :, g, :], dtype=np.float64)
            for hi in his:
                for r0 in range(0, R, chunk):
                    rr = rows[r0:r0 + chunk]
                    if causal:
                        allowed = keys[None, :] <= rr[:, None]
                    else:
                        allowed = np.ones((len(rr), N), dtype=bool)
                    qr = np.asarray(q_rows[b, r0:r0 + len(rr), hi, :], dtype=np.float64)
                    o, lse = attend_rows(qr, K, V, allowed, scale)
                    O[b, r0:r0 + len(rr), hi, :] = o
                    LSE[b, hi, r0:r0 + len(rr)] = lse
    return O, LSE


def attention_weights(q: np.ndarray, k: np.ndarray, causal: bool,
                      scale: Optional[float] = None):
    """The full attention matrix A [B, H, N, N] (rows sum to 1) for tiny inputs."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, N, H, d = q.shape
    G = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    A = np.zeros((B, H, N, N))
    keys = np.arange(N)
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, G)
            S = (q[b, :, h, :] @ k[b, :, g, :].T) * scale
            if causal:
                S = np.where(keys[None, :] <= keys[:, None], S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            E = np.exp(S - m)
            A[b, h] = E / E.sum(axis=1, keepdims=True)
    return A

"""Gradients of softmax attention, and the backward ring, in fp64 on the CPU.

TEST INFRASTRUCTURE (see oracle/__init__.py): never imported by the product path.

What the backward computes is the derivative of the forward's output O with
respect to Q, K and V, contracted with an upstream gradient dO (the gradient of
some scalar loss with respect to O).  The pages fix the structure, not the
formulas:
  * Transformer Math "Ring Attention" (aicassindra), "The backward pass costs a
    second ring": the gradient of K_j, V_j collects contributions from every
    query block that saw block j, so K/V blocks rotate a second time and their
    accumulated gradients rotate with them, each device adding its local
    contribution as a block passes; the [b, b] score blocks are recomputed, and
    only the output and the per-row statistics (m, l) are kept from the forward.
  * "Ring Attention: what the near-infinite context paper actually says",
    "Production tradeoffs no one mentions in the benchmark post" ("Gradient
    correctness requires explicit verification"): gradients with respect to Q,
    K and V flow back through the ring in the reverse direction, and must match
    a single-device reference.

The formulas are the chain rule through S = scale * Q K^T (masked), A = softmax
over each row's admitted keys, O = A V (derived here; the pages print none):
    dV = A^T dO
    dA = dO V^T
    dS = A * (dA - rowsum(A * dA))          (softmax Jacobian, row by row)
    dQ = scale * dS K
    dK = scale * dS^T Q
Masked entries have A = 0 and so dS = 0.  With grouped-query attention the
gradient of kv head g sums over the query heads that read it.

Readings where the pages are silent:
  * The kept statistics (m, l) enter only through LSE = m + ln l, since
    exp(S - m) / l = exp(S - LSE); the ring backward takes LSE.
  * rowsum(A * dA) = rowsum(dO * O) for every row (because O = A V), so the
    ring backward forms D = rowsum(dO * O) from the saved output once per row,
    as the pages keep the output for that purpose; the dense reference uses
    rowsum(A * dA) directly, and the tests check the two agree.
  * "Reverse direction": at backward step s = 0 .. P-1, device u holds the
    circulating K/V block (u + s) mod P together with its dK/dV, i.e. block b
    meets query shards u = (b - s) mod P (the forward had b = (u - s) mod P).
    The direction only changes the summation order.
  * A row that admits no key (LSE = -inf) contributes nothing.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence

import numpy as np

from .attention import default_scale, kv_head_of
from .shardmap import shard_tokens


def _softmax_rows(S: np.ndarray) -> np.ndarray:
    """Row softmax of scaled scores with -inf on masked keys; an all-masked row is 0."""
    m = S.max(axis=1, keepdims=True) if S.shape[1] else np.full((S.shape[0], 1), -np.inf)
    live = np.isfinite(m)
    E = np.exp(S - np.where(live, m, 0.0))
    E = np.where(live, E, 0.0)
    z = E.sum(axis=1, keepdims=True)
    return E / np.where(z > 0, z, 1.0)


def row_block_grads(qr: np.ndarray, K: np.ndarray, V: np.ndarray, dor: np.ndarray,
                    allowed: np.ndarray, scale: float):
    """Chain rule for a block of query rows against all of their keys.

    qr, dor [R, d]: query rows and their upstream gradients; K, V [Nk, d];
    allowed [R, Nk] the mask.  Every admitted key of each row must be among K
    (the softmax is over these keys).  Returns (dq [R, d], dk [Nk, d],
    dv [Nk, d]) -- dk and dv are these rows' contributions only.
    """
    S = np.where(allowed, (qr @ K.T) * scale, -np.inf)
    A = _softmax_rows(S)
    dA = dor @ V.T
    Dr = (A * dA).sum(axis=1, keepdims=True)
    dS = A * (dA - Dr)
    return scale * (dS @ K), scale * (dS.T @ qr), A.T @ dor


def _mask(q_pos, k_pos, causal: bool) -> np.ndarray:
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    if causal:
        return k_pos[None, :] <= q_pos[:, None]
    return np.ones((len(q_pos), len(k_pos)), dtype=bool)


def attention_grads(q, k, v, do, causal: bool, scale: Optional[float] = None,
                    max_chunk_elems: int = 1 << 22):
    """dQ, dK, dV of dense softmax attention for upstream gradient dO.

    q, do [B, N, H, d]; k, v [B, N, G, d]; any float dtype (converted to fp64).
    Returns dq [B, N, H, d], dk, dv [B, N, G, d] in fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, N, H, d = q.shape
    G = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pos = np.arange(N)
    chunk = max(1, max_chunk_elems // max(N, 1))
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, G)
            K, V = k[b, :, g], v[b, :, g]
            for r0 in range(0, N, chunk):
                rr = pos[r0:r0 + chunk]
                a, bk, bv = row_block_grads(q[b, rr, h], K, V, do[b, rr, h],
                                            _mask(rr, pos, causal), scale)
                dq[b, rr, h] = a
                dk[b, :, g] += bk
                dv[b, :, g] += bv
    return dq, dk, dv


def query_grads_at(rows: Sequence[int], heads: Sequence[int], q, k, v, do, causal: bool,
                   scale: Optional[float] = None):
    """dQ of the given query tokens (original order) and heads only: each row
    needs nothing but its own scores against all keys.  Returns [B, R, Hs, d]."""
    B, N, H, d = q.shape
    G = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((B, len(rows), len(heads), d))
    pos = np.arange(N)
    for b in range(B):
        for hi, h in enumerate(heads):
            g = kv_head_of(h, H, G)
            K = np.asarray(k[b, :, g], dtype=np.float64)
            V = np.asarray(v[b, :, g], dtype=np.float64)
            qr = np.asarray(q[b, rows, h], dtype=np.float64)
            dor = np.asarray(do[b, rows, h], dtype=np.float64)
            a, _, _ = row_block_grads(qr, K, V, dor, _mask(rows, pos, causal), scale)
            out[b, :, hi] = a
    return out


def key_grads_at(keys: Sequence[int], q, k, v, do, causal: bool, scale: Optional[float] = None,
                 rows_per_chunk: int = 256):
    """dK and dV of the given key tokens (original order), for every kv head.

    Sums over every query row that admits one of the keys (under the causal
    mask: rows at or after the key); each such row's softmax runs over all of
    its own keys.  Returns dk, dv [B, len(keys), G, d]."""
    B, N, H, d = q.shape
    G = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    keys = np.asarray(keys, dtype=np.int64)
    dk = np.zeros((B, len(keys), G, d))
    dv = np.zeros((B, len(keys), G, d))
    pos = np.arange(N)
    first = int(keys.min()) if causal else 0
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, G)
            K = np.asarray(k[b, :, g], dtype=np.float64)
            V = np.asarray(v[b, :, g], dtype=np.float64)
            for r0 in range(first, N, rows_per_chunk):
                rr = pos[r0:r0 + rows_per_chunk]
                n_keys = int(rr[-1]) + 1 if causal else N   # keys any of these rows may see
                qr = np.asarray(q[b, rr, h], dtype=np.float64)
                dor = np.asarray(do[b, rr, h], dtype=np.float64)
                _, bk, bv = row_block_grads(qr, K[:n_keys], V[:n_keys], dor,
                                            _mask(rr, pos[:n_keys], causal), scale)
                sel = keys < n_keys
                dk[b, sel, g] += bk[keys[sel]]
                dv[b, sel, g] += bv[keys[sel]]
    return dk, dv


def backward_ring_order(b: int, P: int):
    """Query shards that circulating K/V block b meets at backward steps
    s = 0 .. P-1 when the ring runs in the reverse direction: u = (b - s) mod P
    (device u holds block (u + s) mod P at step s)."""
    return [(b - s) % P for s in range(P)]


def ring_backward(q, k, v, o, lse, do, P: int, layout: str, causal: bool,
                  scale: Optional[float] = None,
                  order: Optional[Callable[[int], Sequence[int]]] = None,
                  trace: Optional[Callable[[int, int, int, int, int], None]] = None):
    """The backward ring over P virtual shards.

    q, o, do [B, N, H, d]; k, v [B, N, G, d]; lse [B, H, N] (natural log), as
    saved by the forward.  For every circulating K/V block b, in the order
    order(b) (default: the reverse ring), the query shard u it meets recomputes
    its scores against the block and adds its contributions:
        S   = scale * Q_u K_b^T  (causal mask on global positions)
        A   = exp(S - LSE_u)      (rows with LSE = -inf: 0)
        dV_b += A^T dO_u
        dS  = A * (dO_u V_b^T - D_u),  D_u = rowsum(dO_u * O_u)
        dQ_u += scale * dS K_b
        dK_b += scale * dS^T Q_u
    trace(bi, h, b, s, u) is called after every block visit.  Returns dq, dk,
    dv in original token order, fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    B, N, H, d = q.shape
    G = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    order = order or (lambda b: backward_ring_order(b, P))
    toks = [np.asarray(shard_tokens(layout, N, P, u)) for u in range(P)]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = (do * o).sum(axis=3)                          # [B, N, H]
    for bi in range(B):
        for h in range(H):
            g = kv_head_of(h, H, G)
            for b in range(P):
                tk = toks[b]
                Kb, Vb = k[bi, tk, g], v[bi, tk, g]
                dKb = np.zeros_like(Kb)
                dVb = np.zeros_like(Vb)
                visits = list(order(b))
                assert sorted(visits) == list(range(P)), "every query shard exactly once"
                for s, u in enumerate(visits):
                    tq = toks[u]
                    S = (q[bi, tq, h] @ Kb.T) * scale
                    allowed = _mask(tq, tk, causal)
                    L = lse[bi, h, tq][:, None]
                    live = np.isfinite(L)
                    A = np.where(allowed & live, np.exp(np.where(allowed, S, 0.0)
                                                        - np.where(live, L, 0.0)), 0.0)
                    dVb += A.T @ do[bi, tq, h]
                    dS = A * (do[bi, tq, h] @ Vb.T - D[bi, tq, h][:, None])
                    dq[bi, tq, h] += scale * (dS @ Kb)
                    dKb += scale * (dS.T @ q[bi, tq, h])
                    if trace is not None:
                        trace(bi, h, b, s, u)
                dk[bi, tk, g] += dKb
                dv[bi, tk, g] += dVb
    return dq, dk, dv

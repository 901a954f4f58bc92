"""The ring recurrence over P virtual shards, in fp64 on the CPU.

TEST INFRASTRUCTURE (see oracle/__init__.py): never imported by the product path.

Follows "Ring Attention" (aarnphm.xyz), the ring recurrence display: device u
keeps its query shard; at ring step s it scores its queries against the
circulating shard b(u, s) = (u - s) mod p,
    S     = Q_u K_b^T / sqrt(d_h)
    m_new = max(m_old, max_j S_j)
    z_new = z_old * exp(m_old - m_new) + sum_j exp(S_j - m_new)
    y_new = y_old * exp(m_old - m_new) + sum_j exp(S_j - m_new) V_j
and after all p shards O = y / z.  The same update, with (m, l, acc), is
"Building block: the online-softmax trick" in "Ring Attention: Distributed
Attention Across Devices" (aicomputerinstitute), and (m, l, o) in "Part 4: Ring
Attention" (Fofadiya) 4.4.

Readings where the pages are silent:
  * Steps run s = 0 .. P-1 and step 0 is the local shard (the chapter's worked
    example and "Part 4" 4.3.2); the aarnphm display counts from 1 -- both visit
    every shard once.
  * Initial state m = -inf, z = 0, y = 0 (the chapter's worked example).  When
    nothing was accumulated (m_old = -inf) the old state is zero, so the rescale
    factor is irrelevant and taken as 0; when a block admits no key for a row
    and nothing was accumulated (m_new = -inf) the row state stays unchanged.
  * y is the *unnormalised* running output; it is divided by z once, at the end.
  * LSE = m + ln z.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

import numpy as np

from .attention import default_scale, kv_head_of
from .shardmap import shard_tokens


class RowState:
    """Running (m, z, y) for a set of query rows."""

    def __init__(self, rows: int, d: int):
        self.m = np.full(rows, -np.inf)
        self.z = np.zeros(rows)
        self.y = np.zeros((rows, d))

    def copy(self) -> "RowState":
        c = RowState(0, 0)
        c.m, c.z, c.y = self.m.copy(), self.z.copy(), self.y.copy()
        return c


def fold(state: RowState, S: np.ndarray, V: np.ndarray) -> RowState:
    """Fold one block of scaled scores S [rows, keys] (masked keys = -inf) and
    its values V [keys, d] into the running state, in place."""
    blk_max = S.max(axis=1) if S.shape[1] > 0 else np.full(S.shape[0], -np.inf)
    m_new = np.maximum(state.m, blk_max)
    live = np.isfinite(m_new)                       # rows that have seen a key
    had = np.isfinite(state.m)
    both = had & live
    diff = np.where(both, state.m - np.where(both, m_new, 0.0), 0.0)
    alpha = np.where(both, np.exp(diff), 0.0)
    alpha = np.where(live, alpha, 1.0)              # nothing seen yet: keep the state
    m_ref = np.where(live, m_new, 0.0)
    E = np.exp(S - m_ref[:, None])                  # exp(-inf) = 0 on masked keys
    E = np.where(live[:, None], E, 0.0)
    state.z = alpha * state.z + E.sum(axis=1)
    state.y = alpha[:, None] * state.y + E @ V
    state.m = np.where(live, m_new, state.m)
    return state


def finalize(state: RowState):
    """O = y / z and LSE = m + ln z; a row that saw no key gives O = 0, LSE = -inf."""
    seen = state.z > 0
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(seen[:, None], state.y / np.where(seen, state.z, 1.0)[:, None], 0.0)
        lse = np.where(seen, state.m + np.log(np.where(seen, state.z, 1.0)), -np.inf)
    return O, lse


def ring_order(u: int, P: int) -> List[int]:
    """Shards visited by device u at steps s = 0 .. P-1: b = (u - s) mod P."""
    return [(u - s) % P for s in range(P)]


def scores_block(q_rows: np.ndarray, K: np.ndarray, scale: float, q_pos: Sequence[int],
                 k_pos: Sequence[int], causal: bool) -> np.ndarray:
    """S = scale * Q K^T with keys after the query position set to -inf."""
    S = (q_rows @ K.T) * scale
    if causal:
        qp = np.asarray(q_pos)[:, None]
        kp = np.asarray(k_pos)[None, :]
        S = np.where(kp <= qp, S, -np.inf)
    return S


def ring_attention(q, k, v, P: int, layout: str, causal: bool, scale: Optional[float] = None,
                   order: Optional[Callable[[int], Sequence[int]]] = None,
                   trace: Optional[Callable[[int, int, int, int, int, RowState], None]] = None):
    """Forward ring attention over P virtual shards.

    q [B,N,H,d], k/v [B,N,G,d] (fp64). order(u) gives the shard visit order of
    device u (default: the ring order). trace(b, h, u, s, shard, state) is
    called after every fold. Returns O [B,N,H,d] and LSE [B,H,N] in original
    token order.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, N, H, d = q.shape
    G = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    order = order or (lambda u: ring_order(u, P))
    toks = [np.asarray(shard_tokens(layout, N, P, u)) for u in range(P)]
    O = np.zeros((B, N, H, d))
    LSE = np.zeros((B, H, N))
    for bi in range(B):
        for h in range(H):
            g = kv_head_of(h, H, G)
            for u in range(P):
                tq = toks[u]
                st = RowState(len(tq), d)
                visits = list(order(u))
                assert sorted(visits) == list(range(P)), "every shard exactly once"
                for s, b in enumerate(visits):
                    tk = toks[b]
                    S = scores_block(q[bi, tq, h, :], k[bi, tk, g, :], scale, tq, tk, causal)
                    fold(st, S, v[bi, tk, g, :])
                    if trace is not None:
                        trace(bi, h, u, s, b, st)
                o, lse = finalize(st)
                O[bi, tq, h, :] = o
                LSE[bi, h, tq] = lse
    return O, LSE


def shard_partials(q, k, v, P: int, layout: str, causal: bool, scale: Optional[float] = None):
    """Per-shard normalised partials: for every key shard b, the attention of
    all queries over the keys of shard b alone.

    Returns O_parts [P, B, N, H, d] and LSE_parts [P, B, H, N] (original token
    order; a row that admits no key of shard b has O = 0, LSE = -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, N, H, d = q.shape
    G = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    toks = [np.asarray(shard_tokens(layout, N, P, u)) for u in range(P)]
    Op = np.zeros((P, B, N, H, d))
    Lp = np.zeros((P, B, H, N))
    allq = np.arange(N)
    for bi in range(B):
        for h in range(H):
            g = kv_head_of(h, H, G)
            for b in range(P):
                tk = toks[b]
                st = RowState(N, d)
                S = scores_block(q[bi, :, h, :], k[bi, tk, g, :], scale, allq, tk, causal)
                fold(st, S, v[bi, tk, g, :])
                o, lse = finalize(st)
                Op[b, bi, :, h, :] = o
                Lp[b, bi, h, :] = lse
    return Op, Lp

"""Merge of normalised partial results and finalize of a running state (fp64).

TEST INFRASTRUCTURE (see oracle/__init__.py): never imported by the product path.

Several partial attentions of the same query rows over disjoint key sets combine
by the same rescale-and-add that folds shards in the ring:
  * Transformer Math "Ring Attention" (aicassindra), "The ring is a prefill
    algorithm": each device forms a partial (m, l, o) on its own shard and the
    P triples are combined with one small reduction, the same rescale-and-add.
  * "Ring Attention: what the near-infinite context paper actually says",
    "What the online softmax accumulation actually does across rounds": the
    combination of two partial results with their maxima and sums.
  * "Part 4: Ring Attention" (Fofadiya) 4.9.4.4: partial outputs gathered back
    and combined (pass-Q decode).
A normalised partial carries O_p = y_p / z_p and LSE_p = m_p + ln z_p, so
z_p e^{m_p} = e^{LSE_p}; the merged result is
    LSE = M + ln sum_p e^{LSE_p - M},  M = max_p LSE_p
    O   = sum_p e^{LSE_p - LSE} O_p.
A part with LSE_p = -inf (the row admitted no key there) contributes nothing; if
every part is -inf the row is O = 0, LSE = -inf.
"""
from __future__ import annotations

import numpy as np


def merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """o_parts [n, B, N, H, d], lse_parts [n, B, H, N] -> O [B, N, H, d], LSE [B, H, N]."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = lse_parts.max(axis=0)                                   # [B, H, N]
    dead = ~np.isfinite(M)
    M_safe = np.where(dead, 0.0, M)
    w = np.exp(lse_parts - M_safe[None])                        # e^{-inf} = 0
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(dead, -np.inf, M_safe + np.log(np.where(dead, 1.0, tot)))
        wn = np.where(dead[None], 0.0, w / np.where(dead, 1.0, tot)[None])  # [n, B, H, N]
    # weights to [n, B, N, H, 1] to match o_parts
    wn_t = np.transpose(wn, (0, 1, 3, 2))[..., None]
    O = (wn_t * o_parts).sum(axis=0)
    return O, lse


def finalize(m: np.ndarray, z: np.ndarray, y: np.ndarray):
    """Running state -> result: O = y / z and LSE = m + ln z.

    m, z [B, H, N]; y [B, N, H, d]. A row with z = 0 (no key seen) gives O = 0,
    LSE = -inf. Follows "Ring Attention" (aarnphm.xyz), O = y / z, and "Part 4:
    Ring Attention" 4.4 FINAL (divide the accumulated sum once).
    """
    m = np.asarray(m, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    seen = z > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(seen, m + np.log(np.where(seen, z, 1.0)), -np.inf)
        zt = np.transpose(np.where(seen, z, 1.0), (0, 2, 1))[..., None]   # [B, N, H, 1]
        st = np.transpose(seen, (0, 2, 1))[..., None]
        O = np.where(st, y / zt, 0.0)
    return O, lse

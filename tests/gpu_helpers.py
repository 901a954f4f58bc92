"""Shared helpers of the GPU parity tests: exact host copies of bf16 tensors and
oracle comparisons on full or sampled query rows."""
from __future__ import annotations

import numpy as np
import torch

from oracle import shardmap as OS
from oracle.attention import attention_at, kv_head_of

TOL_O = 1e-2      # max |O_gpu - O_oracle| for bf16 inputs, fp32 accumulation
TOL_LSE = 1e-3    # max |LSE_gpu - LSE_oracle|


def host32(t: torch.Tensor) -> np.ndarray:
    """Exact fp32 host copy of a bf16/fp32 device tensor."""
    return t.detach().float().cpu().numpy()


def edge_rows(layout: str, N: int, P: int, shards=None):
    """First and last local row of each listed shard (default: every shard)."""
    S = N // P
    rows = set()
    for u in (range(P) if shards is None else shards):
        rows.add(OS.token_of(layout, N, P, u, 0))
        rows.add(OS.token_of(layout, N, P, u, S - 1))
    return rows


def sample_rows(layout: str, N: int, P: int, n_random: int, seed: int, shards=None):
    rows = edge_rows(layout, N, P, shards)
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, N, n_random))
    return np.array(sorted(rows), dtype=np.int64)


def compare_rows(o: torch.Tensor, lse: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
                 v: torch.Tensor, causal: bool, rows, heads, scale=None):
    """Max |dO| and |dLSE| of the GPU result against the oracle on the given
    query rows and heads. o, lse, q, k, v may live on the GPU."""
    rows = np.asarray(rows, dtype=np.int64)
    heads = list(heads)
    ridx = torch.as_tensor(rows, device=q.device)
    hidx = torch.as_tensor(heads, device=q.device)
    q_rows = host32(q.index_select(1, ridx).index_select(2, hidx))
    Hn = q.shape[2]
    G = k.shape[2]
    gs = sorted({kv_head_of(h, Hn, G) for h in heads})
    # keep only the kv heads in use, renumbered, to bound host memory
    gidx = torch.as_tensor(gs, device=k.device)
    k_h = host32(k.index_select(2, gidx))
    v_h = host32(v.index_select(2, gidx))
    # map query heads onto the reduced kv-head list: build a virtual head count
    # in which head h reads reduced kv head gs.index(g)
    O_ref = np.zeros((q.shape[0], len(rows), len(heads), q.shape[3]))
    L_ref = np.zeros((q.shape[0], len(heads), len(rows)))
    for gi, g in enumerate(gs):
        his = [i for i, h in enumerate(heads) if kv_head_of(h, Hn, G) == g]
        O_g, L_g = attention_at(q_rows[:, :, his], rows, [0] * len(his), 1,
                                k_h[:, :, gi:gi + 1], v_h[:, :, gi:gi + 1], causal, scale)
        O_ref[:, :, his] = O_g
        L_ref[:, his] = L_g
    o_s = host32(o.index_select(1, ridx).index_select(2, hidx)).astype(np.float64)
    l_s = host32(lse.index_select(1, hidx).index_select(2, ridx)).astype(np.float64)
    eo = float(np.abs(o_s - O_ref).max())
    el = float(np.abs(l_s - L_ref).max())
    return eo, el


def compare_full(o, lse, q, k, v, causal, scale=None):
    N, H = q.shape[1], q.shape[2]
    return compare_rows(o, lse, q, k, v, causal, np.arange(N), range(H), scale)

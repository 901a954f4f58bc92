"""Seeded synthetic inputs for the ring-attention forward path.

This module is the one piece shared by the CUDA path's tests/bench and by the
oracle's tests. It draws random numbers and shapes them; it holds none of the
attention arithmetic (no scores, no softmax, no merge).

Workloads follow the shapes and value distributions of the ring-attention
configurations this library is measured on: i.i.d. N(0, 1) bf16 Q/K/V in
[B, N, heads, d] token-major layout, grouped-query attention with 32 query
heads over 8 KV heads, causal masking, contiguous or striped shard layouts.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

LAYOUTS = ("contiguous", "striped")


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    heads: int
    kv_heads: int
    head_dim: int
    P: int
    layout: str
    causal: bool
    seed: int
    # Multiply Q and K by this factor after drawing (then round to bf16).
    qk_prescale: Optional[float] = None
    # Fraction of token positions per batch whose K rows (all kv heads) are
    # multiplied by `stress_factor` (exact in bf16 for powers of two).
    stress_frac: float = 0.0
    stress_factor: float = 8.0

    @property
    def shard_len(self) -> int:
        return self.seqlen // self.P

    def causal_flops(self) -> float:
        """4*d FLOPs per (q, k) pair per head; causal counts half of N^2."""
        f = 4.0 * self.batch * self.heads * self.seqlen * self.seqlen * self.head_dim
        return f / 2.0 if self.causal else f

    def visible_pairs(self) -> int:
        """Exact number of (query, key) pairs the mask admits, per (batch, head)."""
        n = self.seqlen
        return n * (n + 1) // 2 if self.causal else n * n

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five measured ring-attention configurations (sizes, layouts, distributions).
WORKLOADS = {
    "c1": Workload("c1", 1, 1024, 1, 1, 64, 4, "contiguous", False, 1001),
    "c2": Workload("c2", 1, 32768, 32, 8, 128, 8, "contiguous", True, 1002,
                   qk_prescale=1.0 / math.sqrt(2.0)),
    "c3": Workload("c3", 1, 65536, 32, 8, 128, 16, "striped", True, 1003),
    "c4": Workload("c4", 2, 131072, 32, 8, 128, 16, "contiguous", True, 1004,
                   stress_frac=0.01, stress_factor=8.0),
    "c5": Workload("c5", 1, 1048576, 32, 8, 128, 64, "striped", True, 1005),
}

WORKLOAD_TEXT = {
    "c1": "B=1 N=1024 H=1 G=1 d=64 P=4 contiguous non-causal",
    "c2": "B=1 N=32768 H=32 G=8 d=128 P=8 contiguous causal, Q,K x 1/sqrt(2)",
    "c3": "B=1 N=65536 H=32 G=8 d=128 P=16 striped causal",
    "c4": "B=2 N=131072 H=32 G=8 d=128 P=16 contiguous causal, 1% K rows x8",
    "c5": "B=1 N=1048576 H=32 G=8 d=128 P=64 striped causal",
}


def make_qkv(w: Workload, device="cpu", seed: Optional[int] = None):
    """Draw Q [B,N,H,d], K and V [B,N,G,d] as bf16 from one seeded generator.

    Q, K, V are drawn in that order from N(0, 1) in fp32 and rounded to bf16.
    The stress rows (if any) come from a second generator seeded seed+1.
    """
    seed = w.seed if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    B, N, H, G, d = w.batch, w.seqlen, w.heads, w.kv_heads, w.head_dim

    def draw(shape):
        x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        return x

    q = draw((B, N, H, d))
    k = draw((B, N, G, d))
    v = draw((B, N, G, d))
    if w.qk_prescale is not None:
        q.mul_(w.qk_prescale)
        k.mul_(w.qk_prescale)
    q = q.to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    v = v.to(torch.bfloat16)
    if w.stress_frac > 0.0:
        for b, rows in enumerate(stress_positions(w, seed)):
            rows = rows.to(dev)
            k[b, rows] = k[b, rows] * w.stress_factor
    return q, k, v


def stress_positions(w: Workload, seed: Optional[int] = None):
    """Per batch, the token positions whose K rows make_qkv multiplies by
    stress_factor: the first round(stress_frac * N) entries of a random permutation
    of the N positions, drawn batch after batch from a CPU generator seeded seed+1
    (seed defaults to the workload's). Empty tensors when the workload has none."""
    seed = w.seed if seed is None else seed
    if w.stress_frac <= 0.0:
        return [torch.empty(0, dtype=torch.int64) for _ in range(w.batch)]
    gs = torch.Generator(device="cpu")
    gs.manual_seed(seed + 1)
    n_rows = max(1, int(round(w.stress_frac * w.seqlen)))
    return [torch.randperm(w.seqlen, generator=gs)[:n_rows] for _ in range(w.batch)]


def make_dout(w: Workload, device="cpu", seed: Optional[int] = None):
    """Upstream gradient dO [B,N,H,d] for the backward: N(0, 1) in fp32 rounded to
    bf16, from its own generator seeded seed+2 (seed defaults to the workload's)."""
    seed = w.seed if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 2)
    x = torch.randn((w.batch, w.seqlen, w.heads, w.head_dim), generator=g, device=dev,
                    dtype=torch.float32)
    return x.to(torch.bfloat16)


def make_merge_inputs(n_parts: int, batch: int, seqlen: int, heads: int, head_dim: int,
                      device="cpu", seed: int = 7, neg_inf_frac: float = 0.01):
    """Per-part normalised outputs O_p ~ N(0,1) fp32 [n,B,N,H,d] and log-sum-exps
    LSE_p ~ U(-5, 5) fp32 [n,B,H,N], with a fraction of LSE_p set to -inf
    (a part in which the row saw no key)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    o = torch.randn((n_parts, batch, seqlen, heads, head_dim), generator=g, device=dev,
                    dtype=torch.float32)
    lse = torch.rand((n_parts, batch, heads, seqlen), generator=g, device=dev,
                     dtype=torch.float32) * 10.0 - 5.0
    if neg_inf_frac > 0.0:
        drop = torch.rand(lse.shape, generator=g, device=dev) < neg_inf_frac
        lse = torch.where(drop, torch.full_like(lse, -math.inf), lse)
    return o, lse


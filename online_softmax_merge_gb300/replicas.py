"""Process-group plumbing for running the path as independent replicas, one
process per GPU (launched by torch.distributed.run). The data path has no
collective: each rank runs the whole workload on its own GPU; the ranks only
meet at barriers around the timed region and to take the slowest rank's time.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import torch
import torch.distributed as dist


@dataclass
class RankInfo:
    rank: int
    world: int
    local_rank: int

    @property
    def is_main(self) -> bool:
        return self.rank == 0


def rank_info() -> RankInfo:
    return RankInfo(int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
                    int(os.environ.get("LOCAL_RANK", "0")))


def init(info: RankInfo, backend: str) -> None:
    """Join the process group when launched with more than one rank."""
    if info.world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=info.rank, world_size=info.world)


def barrier(info: RankInfo) -> None:
    if info.world > 1:
        dist.barrier()


def max_over_ranks(info: RankInfo, value: float, device="cpu") -> float:
    """The largest value any rank holds (the slowest rank's time)."""
    if info.world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(info: RankInfo, value: float, device="cpu") -> float:
    if info.world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shutdown(info: RankInfo) -> None:
    if info.world > 1 and dist.is_initialized():
        dist.destroy_process_group()

"""The multi-rank path of the bench (independent replicas; ranks meet only at
barriers and to take the slowest rank's time), run as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from online_softmax_merge_gb300 import replicas
    info = replicas.rank_info()
    replicas.init(info, "gloo")
    replicas.barrier(info)
    slowest = replicas.max_over_ranks(info, 10.0 + rank)
    total = replicas.sum_over_ranks(info, 1.0)
    replicas.barrier(info)
    replicas.shutdown(info)
    out.put((rank, info.is_main, slowest, total))


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, True, 11.0, 2.0), (1, False, 11.0, 2.0)]


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    from online_softmax_merge_gb300 import replicas
    info = replicas.rank_info()
    assert (info.rank, info.world, info.is_main) == (0, 1, True)
    replicas.init(info, "gloo")
    assert replicas.max_over_ranks(info, 3.5) == 3.5

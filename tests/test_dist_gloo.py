"""The N > 1 bench path on CPU: two gloo ranks, barrier + max/sum aggregation."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    from w1_a8_bitlinear_02_b300 import dist as D
    r, w, lr = D.init("gloo")
    D.barrier()
    secs, units = D.aggregate(1.0 + r, 10.0 * (r + 1))
    D.finalize()
    q.put((r, w, lr, secs, units))


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, secs, units) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert secs == 2.0          # slowest rank's time
        assert units == 30.0        # work summed over ranks


def test_single_process_is_identity():
    from w1_a8_bitlinear_02_b300 import dist as D
    assert D.aggregate(1.5, 7.0) == (1.5, 7.0)

"""Process-group helpers for running independent BitLinear workloads on N GPUs.

The forward shards without any exchange: each rank runs its own copy of the
workload on its own GPU (weak scaling), so the only collectives are the
barriers around the timed region and one reduction of the timings:
the job's time is the slowest rank's, its work the sum over ranks.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as tdist


def env_rank_world() -> tuple[int, int, int]:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init(backend: str | None = None) -> tuple[int, int, int]:
    """Join the process group when launched by torchrun (WORLD_SIZE > 1)."""
    rank, world, local = env_rank_world()
    if world > 1 and not tdist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        tdist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world, local


def barrier() -> None:
    if tdist.is_initialized():
        tdist.barrier()


def aggregate(seconds: float, units: float, device=None) -> tuple[float, float]:
    """(max seconds over ranks, sum of units over ranks)."""
    if not tdist.is_initialized():
        return float(seconds), float(units)
    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    tdist.all_reduce(u, op=tdist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def finalize() -> None:
    if tdist.is_initialized():
        tdist.destroy_process_group()

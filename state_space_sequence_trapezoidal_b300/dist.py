"""Host-side helpers for running the benchmark as independent replicas on several GPUs.

The SSM core shards by (batch row, head) with no exchange between shards, so a
multi-GPU run is N replicas: each rank draws its own inputs (seeded by rank),
runs the same launches on its own GPU, and the only collectives are a barrier
around the timed region and a max over the ranks' times.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_rank() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) from the torchrun environment (defaults: single process)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init(backend: str) -> tuple[int, int, int]:
    rank, world, local = env_rank()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world, local


def rank_seed(base: int, rank: int) -> int:
    """Seed of a rank's inputs: replicas draw independent batches."""
    return base + 7919 * rank


def barrier() -> None:
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar over all ranks (the slowest rank's time)."""
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput of a weak-scaling run: all ranks' units over the slowest time."""
    return units_per_rank * world / max_seconds

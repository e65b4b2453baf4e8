"""Host-side logic of multi-GPU runs (weak scaling, no data-path collective).

(sequence, value head) units of the GDN-2 prefill are independent, so every
rank runs its own batch and only the timing is reduced: the job's time is the
slowest rank's, and the aggregate throughput counts every rank's tokens.
"""
from __future__ import annotations

import os

import torch


def rank_world():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s batch: distinct per rank, identical across runs."""
    return int(base_seed) + 1000 * int(rank)


def max_over_ranks(value: float, device="cpu") -> float:
    """Maximum of a per-rank float over the default process group (identity
    when torch.distributed is not initialised)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(tokens_per_rank: int, world: int, slowest_ms: float) -> float:
    """Whole-job tokens/s of a weak-scaling run."""
    return world * tokens_per_rank / (slowest_ms * 1e-3)

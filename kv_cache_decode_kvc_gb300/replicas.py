"""Host-side logic for running the decode step as independent replicas, one process per GPU.

The decode step partitions by (sequence, KV head) and has no exchange step, so N GPUs run N
replicas, each decoding its own batch of the same shape (weak scaling).  torch.distributed is
used only for the barrier around the timed region and for taking the slowest rank's time;
nothing on the data path crosses ranks."""
from __future__ import annotations

import os

SEED_STRIDE = 7919  # prime spacing of the replicas' generator seeds


def env_rank():
    """(rank, local_rank, world_size) from the launcher's environment (1 process if unset)."""
    def get(k, d):
        try:
            return int(os.environ.get(k, d))
        except ValueError:
            return d
    return get("RANK", 0), get("LOCAL_RANK", 0), get("WORLD_SIZE", 1)


def replica_seed(seed: int, rank: int) -> int:
    """Generator seed of a replica's K/V/q data: every rank decodes different values of the
    same shape (the lengths stay those of the workload, so every rank does equal work)."""
    return seed + SEED_STRIDE * rank


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over all ranks (the whole job ends when its slowest rank does)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, bytes_per_step_per_rank: float, ms_per_step: float) -> float:
    """GB/s of the whole job: the bytes all ranks processed per step over the slowest rank's
    step time."""
    return world * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9

"""Replica bookkeeping for running the decode step on several GPUs at once.

The decode path shards by (sequence, kv head) with no exchange between shards, and each
process drives one GPU: every rank decodes its own independent sequence ("replicas only",
weak scaling).  The only cross-rank operations are host-side: a barrier around the timed
region and the maximum of the ranks' step times (the step is done when the slowest rank
is).  Nothing here touches the data path.
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class RankInfo:
    rank: int
    world: int
    local: int


def rank_info() -> RankInfo:
    """This process's rank, world size and local rank, from the launcher's environment
    (single process when unset)."""
    return RankInfo(int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
                    int(os.environ.get("LOCAL_RANK", "0")))


def workload_seed(rank: int) -> int:
    """Seed of the sequence a rank decodes: distinct per rank, so replicas do not share
    inputs."""
    return int(rank)


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of `x` over all ranks (the value itself on one rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_bytes_per_second(bytes_per_step_per_rank: float, world: int, step_seconds: float) -> float:
    """Whole-job throughput: every rank moves its own step's bytes within the (max over
    ranks) step time."""
    return world * bytes_per_step_per_rank / step_seconds

"""Host-side bookkeeping for running the operator as independent replicas, one process per GPU.

Heads are independent (Multi-Head Relation builds every head's relation field from that head's
own coordinates, "Ask Self, Ask Others", Sec. 3.2 and Appendix A.2.1), so ranks exchange no data:
each rank runs its own batch of heads and the only collective is the timing reduction below.
The job's time is the slowest rank's; the job's throughput is the units that every rank
processed divided by that time.  Nothing here touches a kernel.
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class Ranks:
    world: int
    rank: int
    local: int

    @property
    def distributed(self) -> bool:
        return self.world > 1


def from_env(env=None) -> Ranks:
    """Rank layout from the launcher's environment (WORLD_SIZE, RANK, LOCAL_RANK); one process
    without a launcher is world 1, rank 0."""
    env = os.environ if env is None else env
    world = int(env.get("WORLD_SIZE", "1"))
    rank = int(env.get("RANK", "0"))
    local = int(env.get("LOCAL_RANK", str(rank)))
    if world < 1 or not 0 <= rank < world or local < 0:
        raise ValueError(f"inconsistent rank layout: WORLD_SIZE={world} RANK={rank} LOCAL_RANK={local}")
    return Ranks(world, rank, local)


def init(ranks: Ranks, backend: str) -> None:
    """Join the process group (no-op for a single process).  The address comes from MASTER_ADDR /
    MASTER_PORT as the launcher sets them."""
    if ranks.distributed:
        import torch.distributed as dist
        dist.init_process_group(backend, rank=ranks.rank, world_size=ranks.world)


def barrier(ranks: Ranks) -> None:
    if ranks.distributed:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ranks: Ranks, value: float, device="cpu") -> float:
    """The largest of every rank's value, known to every rank (a device tensor for NCCL, a host
    tensor for gloo)."""
    if not ranks.distributed:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ranks: Ranks, units_per_rank: float, slowest_seconds: float) -> float:
    """Whole-job throughput: every rank processed ``units_per_rank`` (weak scaling) and the job
    lasted as long as its slowest rank."""
    if slowest_seconds <= 0:
        raise ValueError("the timed region must have a positive duration")
    return ranks.world * units_per_rank / slowest_seconds


def finish(ranks: Ranks) -> None:
    if ranks.distributed:
        import torch.distributed as dist
        dist.destroy_process_group()

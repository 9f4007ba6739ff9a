"""Running the step as independent replicas on the GPUs of one node.

Every sequence's draft + verify step is independent of every other sequence's and the
drafter weights are read-only, so N GPUs run N replicas, one process per GPU, each on
its own batch of sequences; no collective sits on the data path.  The only exchanges
are host bookkeeping around the timed region: a barrier on both sides of it and the
maximum of the ranks' elapsed times, from which the job's aggregate throughput follows
(units all ranks processed / slowest rank's time).
"""
from __future__ import annotations

import dataclasses
import os
from dataclasses import dataclass

# rank r's sequences come from their own stream seed, so no two replicas draft the same
# batch; the weights (the workload's seed) are the same on every rank
SEED_STRIDE = 7919


@dataclass(frozen=True)
class Replica:
    rank: int = 0
    world: int = 1
    local: int = 0

    @property
    def distributed(self) -> bool:
        return self.world > 1


def from_env(env=None) -> Replica:
    """Rank, world size and local rank as a torchrun-style launcher sets them."""
    env = os.environ if env is None else env
    r = Replica(int(env.get("RANK", "0")), int(env.get("WORLD_SIZE", "1")),
                int(env.get("LOCAL_RANK", "0")))
    if not (0 <= r.rank < r.world) or r.local < 0:
        raise ValueError(f"bad replica coordinates {r}")
    return r


def shard(workload, rank: int):
    """The workload rank `rank` runs: the same shapes and weights, its own batch of
    sequences (context features, lengths, verify logits and uniforms)."""
    if rank == 0:
        return workload
    return dataclasses.replace(workload, seq_seed=workload.sseed + SEED_STRIDE * rank)


def barrier(rep: Replica) -> None:
    if rep.distributed:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(rep: Replica, seconds: float, device="cpu") -> float:
    """The largest of the ranks' elapsed times (every rank gets it)."""
    if not rep.distributed:
        return float(seconds)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, rep: Replica, slowest_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest time."""
    if slowest_seconds <= 0:
        raise ValueError("elapsed time must be positive")
    return units_per_rank * rep.world / slowest_seconds

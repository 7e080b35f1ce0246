"""One replica of the workload per GPU, one process per GPU (torchrun).

MALA's (batch, head) units are independent, and the paper's own parallel
layout (tensor parallelism over attention heads) needs no exchange inside
attention.  So several GPUs run independent replicas of the same step: each
rank draws its own seeded inputs and runs the whole path alone; the ranks
agree only on timing, through a barrier on both sides of the timed region
and the maximum of the per-rank times.  Rank 0 alone reports.
"""
from __future__ import annotations

import os


def rank_env() -> tuple[int, int, int]:
    """(rank, world size, local rank) from the torchrun environment; (0, 1, 0)
    when the process was started alone."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(base: int, rank: int) -> int:
    """Seed of rank `rank`'s inputs: distinct per rank, the base seed on rank 0."""
    return base + rank


class Ranks:
    """Barrier and max-over-ranks for a process group (or a single process).

    `dist` is `torch.distributed` with an initialised group, or None for one
    process; `device` is where the reduction tensor lives (the rank's GPU with
    NCCL, the CPU with gloo); `sync` drains the rank's own device work (e.g.
    `torch.cuda.synchronize`) and runs before and after the group barrier.
    """

    def __init__(self, dist=None, device=None, sync=None):
        self.dist = dist
        self.device = device
        self.sync = sync or (lambda: None)
        self.rank = dist.get_rank() if dist is not None else 0
        self.world = dist.get_world_size() if dist is not None else 1

    def barrier(self) -> None:
        self.sync()
        if self.dist is not None:
            self.dist.barrier()
            self.sync()

    def max(self, x: float) -> float:
        """The largest of the ranks' values of `x` (every rank gets it)."""
        if self.dist is None:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    @property
    def reports(self) -> bool:
        """Whether this rank prints the result line."""
        return self.rank == 0

"""Independent training replicas, one process per GPU.

The training step has no exchange between GPUs here: each rank trains its own
copy of the model on its own token stream (weak scaling, no collective on the
data path).  The process group is used only around the timed region: a
barrier before and after it, and a max over ranks of the elapsed time, so that
whole-job throughput is the tokens every rank processed divided by the slowest
rank's time.
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class RankInfo:
    world: int
    rank: int
    local: int


def rank_env(env=None) -> RankInfo:
    """WORLD_SIZE / RANK / LOCAL_RANK as set by torch.distributed.run (1/0/0 without it)."""
    env = os.environ if env is None else env
    return RankInfo(int(env.get("WORLD_SIZE", "1")), int(env.get("RANK", "0")),
                    int(env.get("LOCAL_RANK", "0")))


def token_seed(base_seed: int, rank: int) -> int:
    """Seed of a rank's token stream: rank 0 draws the single-GPU stream, every
    other rank an independent one."""
    return base_seed + 7919 * rank


class Group:
    """The timing collectives of a replica job; a no-op for one process.

    `dist` is torch.distributed after init_process_group (or None), `device`
    the device the reduction tensor lives on (a CUDA device under NCCL, the CPU
    under gloo), `sync` an optional callable run after each barrier (the CUDA
    device synchronise around the timed region)."""

    def __init__(self, dist=None, device="cpu", sync=None):
        self.dist = dist
        self.device = device
        self.sync = sync

    @property
    def world(self) -> int:
        return self.dist.get_world_size() if self.dist is not None else 1

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()
        if self.sync is not None:
            self.sync()

    def max(self, x: float) -> float:
        if self.dist is None:
            return float(x)
        import torch

        t = torch.tensor([float(x)], device=self.device, dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())


def job_throughput(world: int, tokens_per_rank_step: int, steps: int, seconds: float) -> float:
    """Whole-job tokens per second: every rank's tokens over the slowest rank's time."""
    if seconds <= 0:
        raise ValueError("elapsed time must be positive")
    return world * tokens_per_rank_step * steps / seconds

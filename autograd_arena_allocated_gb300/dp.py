"""Data parallelism over the batch: one process per GPU, each running the
training step on its own B/N sequences, then one gradient exchange before
the AdamW update.

The step's loss is the mean token cross entropy over its B*T positions
(tinytorch page, 三.7), so for N equal shards of the batch the full batch's
gradient is the mean of the N shards' gradients.  The parameters, their
gradients and the AdamW moments are flat vectors (one fixed parameter order),
which makes the exchange a collective over one contiguous fp32 buffer.  Two
forms:

* all-reduce: each rank sums the gradient over the ranks in buckets of whole
  parameter tensors (issued last layer first, the order a backward produces
  them), scales it by 1/N, and runs AdamW over the whole vector; every rank
  then holds the same master weights, moments and 16-bit compute copy.
* sharded: a reduce-scatter leaves rank r with the summed slice r of the
  gradient only; AdamW updates that slice of the master weights, whose
  moments only rank r keeps; an all-gather of the updated 16-bit compute
  copy gives every rank the full copy for its next step.

Slices are equal, contiguous and 8-element aligned (the 16-bit copy's slices
start on 16-byte boundaries, as the update kernel's vector loads want): the
flat vectors are padded to a multiple of 8 * N elements, the padding's
gradient is zero and its parameters are never read by the step.

The collectives are torch.distributed calls on the process group the caller
set up (NCCL between GPUs, gloo on CPU tensors); the update is the native
AdamW (tt_adamw) unless another callable is passed.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence, Tuple

ALIGN = 8  # elements: a slice of the 16-bit copy starts on a 16-byte boundary


def padded_length(n: int, world: int, align: int = ALIGN) -> int:
    """Smallest length >= n that splits into `world` equal, `align`-aligned slices."""
    if n <= 0 or world <= 0:
        raise ValueError("n and world must be positive")
    q = align * world
    return (n + q - 1) // q * q


def shard_range(n_pad: int, world: int, rank: int) -> Tuple[int, int]:
    """[lo, hi) of rank's slice of a vector padded by padded_length."""
    if not 0 <= rank < world or n_pad % world:
        raise ValueError("bad rank or unpadded length")
    s = n_pad // world
    return rank * s, (rank + 1) * s


def tensor_buckets(boundaries: Sequence[int], n_pad: int, max_elems: int) -> List[Tuple[int, int]]:
    """Contiguous [lo, hi) buckets of whole parameter tensors, each holding at
    most max_elems elements unless one tensor alone is larger, listed from the
    end of the flat vector to its start (the order in which a backward pass
    finishes the layers' gradients).  `boundaries` are the tensors' start
    offsets in increasing order (the first is 0); the last bucket ends at
    n_pad, so the padding travels with the last tensor."""
    if not boundaries or boundaries[0] != 0 or list(boundaries) != sorted(boundaries):
        raise ValueError("boundaries must start at 0 and increase")
    ends = list(boundaries[1:]) + [n_pad]
    out: List[Tuple[int, int]] = []
    hi = n_pad
    lo = hi
    for start, end in zip(reversed(boundaries), reversed(ends)):
        if hi - start > max_elems and lo < hi:
            out.append((lo, hi))
            hi = lo
        lo = start
    if lo < hi:
        out.append((lo, hi))
    return out


def tensor_starts(cfg) -> List[int]:
    """Start offsets of the parameter tensors in the flat vector of a model
    configuration (api.make_config), in increasing order."""
    from . import api

    starts = [api.param_offset(cfg, 0, 0)[0], api.param_offset(cfg, 0, 1)[0]]
    for layer in range(cfg.L):
        starts += [api.param_offset(cfg, layer, 2 + j)[0] for j in range(12)]
    return starts + [api.param_offset(cfg, 0, 14)[0], api.param_offset(cfg, 0, 15)[0]]


@dataclass
class Hyper:
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float


# update(master, lowp, grads, m, v, hyper, step) on matching slices
Update = Callable[..., None]


def native_update(ctx) -> Update:
    """The native fused AdamW of a context (tt_adamw) as an update callable."""
    def run(master, lowp, grads, m, v, h: Hyper, step: int):
        ctx.adamw(master, lowp, grads, m, v, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, step)
    return run


class DataParallel:
    """The gradient exchange of one rank.

    `dist` is torch.distributed after init_process_group, `n` the number of
    parameters, `boundaries` the parameter tensors' start offsets (for the
    all-reduce buckets; None = one bucket)."""

    def __init__(self, dist, n: int, boundaries: Optional[Sequence[int]] = None,
                 bucket_elems: int = 1 << 23):
        self.dist = dist
        self.world = dist.get_world_size()
        self.rank = dist.get_rank()
        self.n = n
        self.n_pad = padded_length(n, self.world)
        self.lo, self.hi = shard_range(self.n_pad, self.world, self.rank)
        self.buckets = tensor_buckets(boundaries if boundaries else [0], self.n_pad, bucket_elems)

    # ---------------------------------------------------------- collectives
    def allreduce_mean(self, grads) -> None:
        """grads [n_pad] fp32, in place: the mean over the ranks."""
        self._check(grads, self.n_pad)
        works = [self.dist.all_reduce(grads[lo:hi], op=self.dist.ReduceOp.SUM, async_op=True)
                 for lo, hi in self.buckets]
        for w in works:
            w.wait()
        grads.mul_(1.0 / self.world)

    def reduce_scatter_mean(self, grads, out) -> None:
        """out [n_pad / world] receives this rank's slice of the mean gradient."""
        self._check(grads, self.n_pad)
        self._check(out, self.hi - self.lo)
        self.dist.reduce_scatter_tensor(out, grads, op=self.dist.ReduceOp.SUM)
        out.mul_(1.0 / self.world)

    def allgather(self, shard, full) -> None:
        """full [n_pad] receives every rank's slice (this rank's is `shard`)."""
        self._check(shard, self.hi - self.lo)
        self._check(full, self.n_pad)
        self.dist.all_gather_into_tensor(full, shard)

    # ---------------------------------------------------------- update steps
    def step_allreduce(self, update: Update, master, lowp, grads, m, v, h: Hyper, step: int) -> None:
        """Mean gradient on every rank, then AdamW over the whole vector."""
        self.allreduce_mean(grads)
        update(master, lowp, grads, m, v, h, step)

    def step_sharded(self, update: Update, master_shard, lowp, grads, grad_shard, m_shard, v_shard,
                     h: Hyper, step: int) -> None:
        """This rank's slice of the mean gradient updates its slice of the
        master weights and moments; the updated 16-bit copy is gathered.
        lowp [n_pad] is the full compute copy (its slice [lo, hi) is written by
        the update, then every slice arrives by the all-gather)."""
        self.reduce_scatter_mean(grads, grad_shard)
        mine = lowp[self.lo:self.hi]
        update(master_shard, mine, grad_shard, m_shard, v_shard, h, step)
        self.allgather(mine.clone(), lowp)

    @staticmethod
    def _check(t, n):
        if t.dim() != 1 or t.numel() != n or not t.is_contiguous():
            raise ValueError(f"expected a contiguous flat tensor of {n} elements, got {tuple(t.shape)}")

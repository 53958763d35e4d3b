"""Data-parallel training step over torch.distributed, one process per GPU.

The batch is split on its first dimension and each rank runs the step on its
rows; the gradients are then summed across ranks and every rank applies the
same update (MuNet, pypi "munet-nn", "Reliability, observability and
scaling": mu.DataParallel splits each batch on dim 0 and averages the
gradients; netcl.online "Architecture: Distributed & Multi-Device
Execution", data_parallel_step: shard the batch, synchronise the gradients,
update; noeira.ai "Neural networks", "Distributed training": DDP).

Each rank's gradient step scales the loss gradient by 1 / global_batch, so
the exchange is a plain SUM all-reduce of the flat fp32 gradient plane (one
contiguous buffer, all layers at once) and of the shard losses; the update
then runs on identical gradients on every rank.  torch.distributed is the
transport (NCCL on GPUs; gloo works too); the library's kernels compute
everything else.
"""
from __future__ import annotations

from typing import Optional, Tuple


def shard_rows(global_batch: int, world: int, rank: int) -> Tuple[int, int]:
    """Rows [start, stop) of a global batch that `rank` of `world` ranks
    takes: contiguous, in rank order, sizes differing by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if global_batch < world:
        raise ValueError(f"a batch of {global_batch} rows cannot give each of {world} ranks a row")
    base, extra = divmod(global_batch, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


class DataParallel:
    """A model replica on this rank and the data-parallel step around it.

    `model` is a neural_net_step_gb300.Model (or any object with the same
    batch / grad_step / grad_tensor / apply_update / read_flat / write_flat
    methods) created with batch = this rank's row count for `global_batch`
    (shard_rows).  Without an initialised process group the step runs on this
    process alone."""

    def __init__(self, model, global_batch: int, group=None):
        import torch.distributed as dist
        self.model = model
        self.global_batch = int(global_batch)
        self.dist = dist if dist.is_available() and dist.is_initialized() else None
        self.group = group
        self.world = self.dist.get_world_size(group) if self.dist else 1
        self.rank = self.dist.get_rank(group) if self.dist else 0
        self.rows = shard_rows(self.global_batch, self.world, self.rank)
        if model.batch != self.rows[1] - self.rows[0]:
            raise ValueError(f"rank {self.rank} takes {self.rows[1] - self.rows[0]} rows; the model's batch is "
                             f"{model.batch}")
        self.grad = model.grad_tensor()

    def broadcast_params(self, src: int = 0) -> None:
        """Give every rank the parameters (and step counter) of rank `src`."""
        if self.world == 1:
            return
        import numpy as np
        import torch
        p, step = self.model.read_flat()
        dev = self.grad.device
        t = torch.from_numpy(np.ascontiguousarray(p)).to(dev)
        s = torch.tensor([step], dtype=torch.int64, device=dev)
        self.dist.broadcast(t, src, group=self.group)
        self.dist.broadcast(s, src, group=self.group)
        self.model.write_flat(t.cpu().numpy(), step=int(s.item()))

    def step(self, x, y, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, loss=None):
        """One data-parallel step on this rank's rows x, y (rows
        self.rows of the global batch).  Returns the global batch loss (a
        device scalar, the same on every rank)."""
        loss = self.model.grad_step(x, y, self.global_batch, loss)
        if self.world > 1:
            # ordered after the gradient step on the current stream; the
            # update, launched on the same stream, follows the sum
            self.dist.all_reduce(self.grad, group=self.group)
            self.dist.all_reduce(loss, group=self.group)
        self.model.apply_update(lr, beta1, beta2, eps, wd)
        return loss

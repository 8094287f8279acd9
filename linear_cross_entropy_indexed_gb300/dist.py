"""Host-side glue for running the fused loss token-sharded across ranks.

Each rank holds all of W and its own rows of H and labels.  The forward is local; a
global mean over valid tokens needs one exchange of two integers and one float
(sum of per-row losses, valid count), the ``num_items_in_batch`` logic of the
Unsloth notes (§4, "n_items").  ``flce_backward`` reads the valid count from
``counts[0]`` on the device, so summing ``counts`` across ranks between the two calls
makes every rank scale its gradient by g / n_valid_global.  dH stays local; dW is
summed by the ordinary data-parallel gradient all-reduce.

Nothing here runs arithmetic of the loss itself; the collectives go through
torch.distributed (NCCL for device tensors, gloo for CPU tensors).

Recipe per step::

    loss_sum, lse, counts, _ = flce_forward(H_r, W, y_r, reduction="sum")
    allreduce_counts_(counts)                    # counts[0] = global valid count
    loss = global_mean_loss(loss_sum, counts)    # all-reduce of the local sums
    dH_r, dW_r = flce_backward(H_r, W, y_r, lse, counts, g, reduction="mean")
    torch.distributed.all_reduce(dW_r)           # data-parallel weight gradient
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_rows(N: int, world: int, rank: int) -> slice:
    """Contiguous row range of `rank`; shard sizes differ by at most one row."""
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    return slice(start, start + base + (1 if rank < extra else 0))


def allreduce_counts_(counts: torch.Tensor, group=None) -> torch.Tensor:
    """In place: counts[0:2] (valid, bad) summed over ranks, counts[2] (device error
    bits) combined with a max so any rank's error stays visible."""
    head = counts[0:2].clone()
    tail = counts[2:3].clone()
    dist.all_reduce(head, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(tail, op=dist.ReduceOp.MAX, group=group)
    counts[0:2].copy_(head)
    counts[2:3].copy_(tail)
    return counts


def global_mean_loss(local_loss_sum: torch.Tensor, counts_global: torch.Tensor, group=None) -> torch.Tensor:
    """Sum of every rank's per-row losses divided once by the global valid count
    (0 when no rank has a valid row)."""
    total = local_loss_sum.detach().to(torch.float64).reshape(1).clone()
    dist.all_reduce(total, op=dist.ReduceOp.SUM, group=group)
    n = counts_global[0].to(torch.float64)
    return torch.where(n > 0, total[0] / torch.clamp(n, min=1), torch.zeros_like(total[0])).to(torch.float32)

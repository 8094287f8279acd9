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

Recipe per step (``data_parallel_step`` runs it)::

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


def data_parallel_step(H, W, labels, grad_out=1.0, ignore_index: int = -100, softcap: float = 0.0, group=None,
                       forward=None, backward=None, reduce_dW: bool = True, timer=None, **backward_kw):
    """One token-sharded forward + backward of this rank's rows (the recipe above).

    Returns (loss, dH, dW, counts): the global mean loss (every rank gets the same
    value), this rank's rows of dH, dW summed over the ranks (this rank's part only when
    reduce_dW is False, for callers whose optimizer reduces gradients itself), and the
    exchanged counts [global valid, global bad, error bits of any rank] for check_counts.
    ``forward`` / ``backward`` default to the library's flce_forward / flce_backward and
    take their arguments.  ``timer``, if given, is a context-manager factory wrapped
    around each collective (the benchmark times them with CUDA events)."""
    if forward is None or backward is None:
        from . import flce_backward, flce_forward
        forward = forward or flce_forward
        backward = backward or flce_backward
    timer = timer or _no_timer
    workspace = backward_kw.pop("workspace", None)
    loss_sum, lse, counts, _ = forward(H, W, labels, ignore_index, softcap, "sum", workspace=workspace)
    with timer("counts"):
        allreduce_counts_(counts, group)
        loss = global_mean_loss(loss_sum, counts, group)
    g = grad_out if torch.is_tensor(grad_out) else torch.tensor([float(grad_out)], dtype=torch.float32,
                                                                 device=counts.device)
    dH, dW = backward(H, W, labels, lse, counts, g, ignore_index, softcap, "mean", workspace=workspace,
                      **backward_kw)
    if reduce_dW and dW is not None:
        with timer("dW"):
            dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=group)
    return loss, dH, dW, counts


class _NoTimer:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def _no_timer(name):
    return _NoTimer()


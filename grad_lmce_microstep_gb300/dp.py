"""Data-parallel host logic around the micro-step library.

Rows (tokens) are independent, so data parallelism shards them: every rank runs
its own micro-steps on its own rows with the same W.  Two exchanges remain, both
on the host side of the library:

1. before the first micro-step, a SUM all-reduce of the valid-target count, so
   that every rank scales its gradients by 1 / (valid targets over all ranks and
   micro-steps) -- the global token-weighted mean;
2. after the last micro-step, a SUM all-reduce of the fp32 dW buffer (and of any
   other parameter gradient the step accumulated, such as ln_f's dgamma and dbeta)
   and of (loss_sum, valid_count).

The pages average gradients across ranks (DDP's AVG) after each rank divided its
micro-batch means by grad_accum_steps ("Multi-GPU calculation of gradients for
accelerated training", section "DDP averages gradients across processes").  That
reproduces the global mean only when every rank and micro-step has the same number
of valid targets; with the scale already carrying 1 / global count, the reduction
here is a SUM, which is right for any counts.  Nothing is reduced between
micro-steps (the pages' no_sync pattern).
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def _active(group) -> bool:
    return dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1


def global_valid_count(local_valid: int, group=None, device=None) -> int:
    """Valid targets summed over all ranks (the local count when not distributed)."""
    t = torch.tensor([int(local_valid)], dtype=torch.int64, device=device)
    if _active(group):
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return int(t.item())


def reduce_step(dW: torch.Tensor, loss_sum: float, valid_count: int, group=None, extra=()):
    """SUM-reduce dW (and every tensor in ``extra``) in place; return the summed (loss_sum, valid_count)."""
    if not _active(group):
        return float(loss_sum), int(valid_count)
    dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=group)
    for t in extra:
        if t is not None:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    scal = torch.tensor([float(loss_sum), float(valid_count)], dtype=torch.float64, device=dW.device)
    dist.all_reduce(scal, op=dist.ReduceOp.SUM, group=group)
    return float(scal[0].item()), int(round(scal[1].item()))


def shard_rows(n_rows: int, rank: int, world: int):
    """Contiguous [start, stop) row range of ``rank``; the first n_rows % world ranks get one more."""
    base, extra = divmod(n_rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)

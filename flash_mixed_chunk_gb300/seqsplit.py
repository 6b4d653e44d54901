"""A causal sequence split over ranks: each rank runs one piece of the
sequences with ``flash_mca_forward_seq`` and needs, as its carried-in state,
the sum of the states of the pieces before it (the exclusive prefix of the
per-rank sums over the ranks, in rank order).  Host-side exchange through
``torch.distributed`` (NCCL on GPUs, gloo on the CPU); the sums are added in
rank order on every rank, so all ranks form the same bits."""
from __future__ import annotations

import torch
import torch.distributed as dist


def exclusive_state_scan(local_sum: torch.Tensor, group=None) -> torch.Tensor:
    """The sum of the lower ranks' ``local_sum`` (zeros on rank 0):
    this rank's ``state_in`` when every rank's piece follows the lower ranks'
    pieces in the sequences."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    local_sum = local_sum.contiguous()
    parts = [torch.empty_like(local_sum) for _ in range(world)]
    dist.all_gather(parts, local_sum, group=group)
    out = torch.zeros_like(local_sum)
    for r in range(rank):
        out += parts[r]
    return out

"""Host-side helpers for running the KDA path on several GPUs, one process per GPU.

Every (b, h) sequence of the KDA forward is independent, so the forward shards over
(b, h) with no exchange between ranks.  The backward shards over the batch the same way,
with one exchange: the gradients of the gate's shared parameters (dA_log per head,
ddt_bias per head and channel) are sums over the batch, so the ranks' partial sums are
added by one all-reduce (sum_param_grads).  The other collectives are the barrier and the
max-over-ranks timing reduction a benchmark needs.
"""
from __future__ import annotations

import os
from typing import Tuple


def env() -> Tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 when absent)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_range(n: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous [begin, end) share of n independent units for `rank` of `world`; the shares
    differ in size by at most one and cover [0, n) exactly once."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of {world}")
    base, extra = divmod(n, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over all ranks of the default process group (identity when the
    group is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def sum_param_grads(grads: dict, names=("dA_log", "ddt_bias")) -> dict:
    """Complete the batch sums of the backward's parameter gradients across ranks.

    With the batch sharded over ranks (each rank calling the backward on its own sequences
    with all heads), `grads[n]` holds the sum over that rank's sequences for n in `names`;
    one all-reduce (sum) per tensor, in place, leaves the whole batch's gradient on every
    rank.  Per-token gradients and dh0 belong to the rank's own sequences and are not
    touched.  Identity without an initialised process group of more than one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return grads
    for n in names:
        t = grads.get(n)
        if t is not None:
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return grads

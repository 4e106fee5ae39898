"""Host side of running the pass on several GPUs (one process per GPU).

Every (sequence, layer, KV head) unit is independent through score ->
select -> compact -> decode, so ranks own disjoint units and exchange
nothing on the data path.  Two things cross ranks:
  * timing: a barrier around the timed region and the maximum of the
    ranks' times;
  * CommitKV Eq. 4's shared index set, when a sequence's layers are split
    across ranks: one index set for all layers and heads needs the sum of
    every unit's scores, so each rank sums its own units
    (kvc_shared_scores) and the partial sums are added across ranks with
    one all-reduce before the per-sequence selection.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch


def layer_shard(n_layers: int, world: int, rank: int) -> Tuple[int, int]:
    """Contiguous layer range [l0, l1) of `rank`: sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank outside the world")
    base, extra = divmod(n_layers, world)
    l0 = rank * base + min(rank, extra)
    return l0, l0 + base + (1 if rank < extra else 0)


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def all_reduce_shared(partial: torch.Tensor, world: int, group: Optional[object] = None) -> torch.Tensor:
    """Adds the ranks' partial per-sequence score sums [B][T] in place (CommitKV
    Eq. 4 across layer shards) and returns the tensor."""
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(partial, op=dist.ReduceOp.SUM, group=group)
    return partial

"""Splitting grouped calls across ranks (one process per GPU).

The groups of a grouped call are independent problems, so the path shards
with no collective on the data path:

* weak scaling (what ``bench.py`` reports): every rank runs its own grouped
  call of the same shapes on its own batch (``rank_seed``);
* expert parallel: one grouped call's groups split across ranks by FLOPs
  (``shard_groups``); each rank computes its groups' C, nothing is exchanged.

Only the timing uses a collective: ``max_over_ranks``.
"""
from __future__ import annotations


def rank_seed(base_seed: int, rank: int) -> int:
    """Data seed of a rank's own batch (rank 0 keeps the base seed)."""
    return base_seed + 1000 * rank


def shard_groups(shapes, world_size: int, rank: int):
    """Indices of the groups rank `rank` owns: longest-processing-time
    assignment by 2*M*N*K, ties to the lower rank, groups kept in their
    original order within a rank.  Empty groups go to rank 0."""
    if world_size < 1 or not 0 <= rank < world_size:
        raise ValueError("bad world_size / rank")
    order = sorted(range(len(shapes)), key=lambda i: -2 * shapes[i][0] * shapes[i][1] * shapes[i][2])
    load = [0] * world_size
    owner = [0] * len(shapes)
    for i in order:
        M, N, K = shapes[i]
        if M == 0:
            owner[i] = 0
            continue
        r = min(range(world_size), key=lambda j: (load[j], j))
        owner[i] = r
        load[r] += 2 * M * N * K
    return [i for i in range(len(shapes)) if owner[i] == rank]


def max_over_ranks(x: float, device=None) -> float:
    """Max of a float over all ranks of the default process group (identity
    without one).  `device` is where the reduction tensor lives (CPU for
    gloo, the rank's GPU for NCCL)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())

"""Data-parallel use of the verifier across GPUs (one process per GPU).

Every sequence is verified independently, so a batch shards over sequences with no
exchange on the data path: each rank runs the library on its own sequences. This module
holds only the host-side bookkeeping: which sequences a rank owns, the seed of a rank's
synthetic batch when every rank verifies a batch of its own (weak scaling), and the two
scalar reductions a timing harness needs (the slowest rank's time, the total work)."""
from __future__ import annotations


def shard_bounds(total: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous [lo, hi) share of `total` sequences for `rank` of `world`; the shares
    differ by at most one sequence and cover 0..total exactly once."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    base, extra = divmod(int(total), world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s own synthetic batch (rank 0 keeps the workload's seed)."""
    return int(base_seed) + 1000 * int(rank)


def _reduce(x: float, world: int, device, op: str) -> float:
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def max_over_ranks(x: float, world: int, device) -> float:
    return _reduce(x, world, device, "max")


def sum_over_ranks(x: float, world: int, device) -> float:
    return _reduce(x, world, device, "sum")

"""One process per GPU: launch-environment helpers for replicated runs.

The attention path partitions into independent (batch, kv-head) units, so
ranks share no data: each rank runs its own batch (weak scaling) or its own
slice of the units (``shard_units``).  The only cross-rank communication is
host-side bookkeeping -- a barrier and a max over ranks for timing -- never
anything on the data path.
"""

from __future__ import annotations

import os

import torch
import torch.distributed as dist


def dist_env():
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend: str = "nccl", device=None) -> bool:
    """Join the process group when launched with more than one rank."""
    world, _, _ = dist_env()
    if world <= 1 or dist.is_initialized():
        return world > 1
    kw = {}
    if backend == "nccl" and device is not None:
        kw["device_id"] = device
    dist.init_process_group(backend, **kw)
    return True


def barrier() -> None:
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of ``x`` over all ranks (identity when running alone)."""
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of a rank's own synthetic batch (independent batches per rank)."""
    return int(base_seed) + 1000003 * int(rank)


def shard_units(n_units: int, rank: int, world: int):
    """Contiguous, disjoint slice [lo, hi) of ``n_units`` independent units for ``rank``."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(int(n_units), int(world))
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def aggregate_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: units every rank processed over the slowest rank's time."""
    return world * units_per_rank / seconds

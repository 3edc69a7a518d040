"""Multi-GPU bookkeeping for the attention path: one process per GPU.

Every (batch, head) of attention is independent in both passes, so the work
shards over heads with no data exchange.  This module holds the rank-side
arithmetic shared by the benchmark and the tests: which heads a rank owns
when a fixed problem is split (strong scaling), the max of a per-rank time,
and the whole-job rate.  No collective touches attention data; the only
collectives are control-plane ones on scalars.
"""
from __future__ import annotations


def head_shard(num_heads: int, world: int, rank: int):
    """Contiguous [lo, hi) range of heads owned by `rank` of `world`.

    Shards differ in size by at most one head; their union is every head and
    they are disjoint.
    """
    if world < 1 or not 0 <= rank < world or num_heads < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(num_heads, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar over the default process group (the value
    itself when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest
    rank's time."""
    if max_seconds <= 0:
        raise ValueError("time must be positive")
    return units_per_rank * world / max_seconds

"""Request sharding across ranks (one process per GPU).

Requests are independent and each one's random stream is keyed on its
global index (the Philox counter takes b + request_offset), so a batch can be
split across ranks with no collective on the data path: a rank verifies its
own requests with request_offset = the global index of its first request, and
the results equal those of the unsharded call.  The only collectives are for
measurement (max of the step time over ranks) and, when a caller wants them,
gathering the outputs.
"""
from __future__ import annotations

import torch


def shard(B: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [lo, hi) share of a global batch of B requests (strong scaling)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    return B * rank // world, B * (rank + 1) // world


def weak_offset(rank: int, per_rank_batch: int) -> int:
    """Global index of a rank's first request when every rank holds its own
    batch of per_rank_batch requests (weak scaling)."""
    return rank * per_rank_batch


def _dist():
    import torch.distributed as dist
    return dist if dist.is_available() and dist.is_initialized() else None


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank float over all ranks (the step time of a job is
    its slowest rank's)."""
    dist = _dist()
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    dist = _dist()
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def gather_rows(local: torch.Tensor) -> torch.Tensor:
    """Concatenate every rank's rows (dim 0, possibly uneven) in rank order."""
    dist = _dist()
    if dist is None:
        return local
    world = dist.get_world_size()
    n = torch.tensor([local.shape[0]], dtype=torch.int64, device=local.device)
    sizes = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(sizes, n)
    m = int(max(int(x.item()) for x in sizes))
    pad = torch.zeros((m,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    pad[:local.shape[0]] = local
    out = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(out, pad)
    return torch.cat([o[:int(s.item())] for o, s in zip(out, sizes)], dim=0)

"""Token-row sharding across GPUs (host logic only).

Depth attention never mixes token positions, so the B*T rows of every
source, output and statistic split across ranks with no exchange: rank r
owns one contiguous row range of every tensor, and no collective touches
the data path.  The only cross-rank step of a measurement is the max of
the ranks' elapsed times.
"""
from __future__ import annotations


def row_range(rows: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous [start, stop) rows of `rank`; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("bad rows / world / rank")
    base, extra = divmod(rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_rows(t, world: int, rank: int):
    """The rank's rows of a [B, T, D] (or [rows, D]) tensor, as a contiguous [rows_r, D] view."""
    flat = t.reshape(-1, t.shape[-1])
    a, b = row_range(flat.shape[0], world, rank)
    return flat[a:b]


def max_over_ranks(value: float, group=None) -> float:
    """Max of a per-rank scalar (elapsed time) over the process group; identity when single."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return float(value)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())

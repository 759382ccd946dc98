"""Host-side helpers for running the loss data-parallel over several GPUs.

Tokens are independent in the forward and in dH, so each rank runs the whole hot
path on its own batch of tokens with no collective on the data path.  Only two
reductions cross ranks: the number of valid tokens of the global batch (so that
every rank divides its "mean" by the same denominator, as KDLoss's
num_batch_labels does) and, outside this library, the sum of dW over ranks that a
data-parallel wrapper performs.  `max_over_ranks` serves the benchmark's timing.
"""
from __future__ import annotations

import os

import torch


def world_from_env():
    """(rank, world_size, local_rank) from the torchrun environment (1 process: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_rows(n_total: int, rank: int, world: int):
    """Contiguous token range [start, stop) of `rank` when n_total tokens are split."""
    base, extra = divmod(n_total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def _dist():
    import torch.distributed as dist
    return dist if dist.is_available() and dist.is_initialized() else None


def global_valid_count(labels: torch.Tensor, ignore_index: int) -> int:
    """Valid tokens summed over all ranks (the shared mean denominator)."""
    local = torch.tensor([int((labels != ignore_index).sum().item())], dtype=torch.int64,
                         device=labels.device if _backend_wants_device() else "cpu")
    d = _dist()
    if d is not None:
        d.all_reduce(local, op=d.ReduceOp.SUM)
    return int(local.item())


def max_over_ranks(value: float, device=None) -> float:
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if _backend_wants_device() else "cpu")
    d = _dist()
    if d is not None:
        d.all_reduce(t, op=d.ReduceOp.MAX)
    return float(t.item())


def _backend_wants_device() -> bool:
    d = _dist()
    return d is not None and d.get_backend() == "nccl"

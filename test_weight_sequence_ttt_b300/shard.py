"""Multi-GPU placement of the TTT inner loop: one process per GPU.

Every (sequence, head) chain is independent, so the work splits across ranks
by chains with no exchange on the data path; the only collectives are the
host-side timing reductions of a benchmark (a barrier and a max / sum over
ranks). Works with any torch.distributed backend (nccl on GPUs, gloo on CPU).
"""
from __future__ import annotations

import os
from typing import Optional, Tuple


def world() -> Tuple[int, int]:
    """(rank, world size) from the torchrun environment (0, 1 when absent)."""
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def chain_slice(rank: int, world_size: int, n_chains: int) -> Tuple[int, int]:
    """Contiguous [start, stop) range of chain indices (beta * H + h) owned by
    ``rank``: the first n % world ranks take one extra chain."""
    if world_size < 1 or not 0 <= rank < world_size:
        raise ValueError("rank %d out of range for world size %d" % (rank, world_size))
    base, extra = divmod(n_chains, world_size)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def init(backend: Optional[str] = None):
    """Initialise the default process group when WORLD_SIZE > 1; returns the
    torch.distributed module, or None for a single process."""
    _, ws = world()
    if ws <= 1:
        return None
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend or ("nccl" if torch.cuda.is_available() else "gloo"))
    return dist


def barrier(dist) -> None:
    if dist is not None:
        dist.barrier()


def _reduce(dist, x: float, op) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(dist, x: float) -> float:
    """Slowest rank's value (a step time), the same on every rank."""
    return x if dist is None else _reduce(dist, x, dist.ReduceOp.MAX)


def sum_over_ranks(dist, x: float) -> float:
    """Whole-job total (tokens processed), the same on every rank."""
    return x if dist is None else _reduce(dist, x, dist.ReduceOp.SUM)

"""Multi-GPU plumbing for the benchmark: one process per GPU, each an independent replica.

The select-and-verify step partitions by request (blocks are independent), so N GPUs run
N replicas, each holding its own copy of the LM head and selector tables and serving its
own batch. There is no collective on the data path; torch.distributed is used only for
the start barrier and the max-over-ranks of the measured time.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def rank_info() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) from the launcher's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend: str | None = None) -> tuple[int, int, int]:
    rank, world, local = rank_info()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    if dist.is_initialized():
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float) -> float:
    """Largest value of x across ranks (the slowest replica sets the job's time)."""
    if not dist.is_initialized():
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float) -> float:
    if not dist.is_initialized():
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_throughput(units_per_rank: float, seconds_per_rank: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return sum_over_ranks(units_per_rank) / max_over_ranks(seconds_per_rank)


def shard(n: int, world: int, rank: int) -> range:
    """Contiguous near-equal share of n independent units for `rank`."""
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def finalize():
    if dist.is_initialized():
        dist.destroy_process_group()

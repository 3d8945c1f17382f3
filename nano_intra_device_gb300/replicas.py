"""Multi-GPU execution of the layer step: independent replicas.

The step has no exchange: every request's tokens depend only on its own K/V
history and on the shared weights ("NanoFlow: Towards Optimal LLM Serving
Throughput", "The Intra-Device Parallelism Mechanism": nano-batches, and so
requests, share no data dependencies).  Splitting one step across GPUs would
need tensor parallelism and its collectives, which this library does not use.
So N GPUs run N replicas: one process per GPU, each with its own copy of the
weights, its own KV cache and its own requests, and no collective on the data
path.  The only cross-process calls are for measurement (a barrier and the
maximum step time).

Launch: ``torchrun --nproc-per-node N ...`` (RANK, WORLD_SIZE, LOCAL_RANK,
MASTER_ADDR/PORT from the environment).
"""
from __future__ import annotations

import os

import torch


def setup(backend: str | None = None):
    """Join the process group when launched with WORLD_SIZE > 1.

    Returns (rank, world, local_rank).  backend defaults to nccl when CUDA is
    available, else gloo.
    """
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if backend is None:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    if not dist.is_initialized():
        dist.init_process_group(backend)
    return dist.get_rank(), dist.get_world_size(), local


def _device():
    import torch.distributed as dist
    return torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all replicas (the job's step time)."""
    if world <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int) -> float:
    """Sum over replicas (tokens processed by the whole job)."""
    if world <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=_device())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard(n: int, rank: int, world: int) -> tuple:
    """Contiguous share [begin, end) of n requests for one replica."""
    base, extra = divmod(n, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def teardown(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()

"""Process-group helpers for running independent chunked-attention problems on
several GPUs (one process per GPU).

The path shards without any data exchange: every (batch entry, key/value
head) problem is independent (its query heads, cache head and dK/dV slice),
so ranks take disjoint sets of problems and only the timing is reduced (a
barrier and a max over ranks).  Works with the nccl backend on GPUs and with
gloo on the CPU.
"""

import os

import torch
import torch.distributed as dist


def rank_env():
    """(rank, local_rank, world_size) from the torchrun environment, or a
    single-process default."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def init(backend):
    rank, _, world = rank_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def shard_units(n_units, rank, world):
    """Contiguous, balanced range [lo, hi) of `n_units` independent problems
    for `rank` of `world`."""
    base, extra = divmod(n_units, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def barrier():
    if dist.is_initialized():
        dist.barrier()


def max_over_ranks(x, device="cpu"):
    """Maximum of a float over all ranks (identity without a process group)."""
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, device="cpu"):
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def finalize():
    if dist.is_initialized():
        dist.destroy_process_group()

"""Multi-GPU use of the layer: independent replicas, host side only.

The routed MoE layer of one prefill chunk needs nothing from any other
chunk, so N GPUs take N different chunks of the prompt (or N independent
prompts), each with its own copy of the expert weights.  There is no
collective on the data path; torch.distributed is used only to start the
ranks, to line them up around a timed region and to take the slowest rank's
time.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def init_from_env(backend: str = "nccl"):
    """(rank, world, local_rank) from the torchrun environment; initialises
    the process group when world > 1 (MASTER_ADDR / MASTER_PORT from env)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def chunk_of_rank(rank: int, world: int) -> int:
    """Chunk index a rank processes in the weak-scaling run: its own."""
    return rank


def chunks_of_rank(n_chunks: int, rank: int, world: int) -> list[int]:
    """Round-robin share of a long prompt's chunks: chunk c goes to rank
    c mod world, so every chunk is processed exactly once."""
    return list(range(rank, n_chunks, world))


def barrier(world: int):
    if world > 1:
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return float(value)
    on_gpu = dist.get_backend() == "nccl"
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if on_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def finalize(world: int):
    if world > 1 and dist.is_initialized():
        dist.destroy_process_group()

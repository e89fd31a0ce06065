"""Host-side helpers for running the layer on several ranks.

Expert parallelism ("expert_map" in the signature of ``FusedMoEPermuteExperts
Unpermute.apply`` on page "vllm.model_executor.layers.fused_moe.modular_kernel";
the rocm_aiter path passes the same map): every rank holds a contiguous block
of the global experts and runs the unchanged single-GPU layer with an
``expert_map`` that sends its own experts to local indices and every other
expert to -1 (dropped).  Summing the ranks' outputs gives the full layer; the
exchange that does that sum (an all-to-all combine or an all-reduce) belongs to
the caller's communication layer, not to this library.

Replica runs (the benchmark launched with one process per GPU) only need the
slowest rank's time, ``replica_max``.
"""
from __future__ import annotations

import numpy as np


def expert_partition(E: int, world: int, rank: int) -> tuple[int, int]:
    """[first, first + count) of the global experts owned by ``rank`` when E
    experts are split into ``world`` contiguous blocks (the first E % world
    ranks own one extra expert)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    if E < 0:
        raise ValueError("E must be >= 0")
    base, extra = divmod(E, world)
    count = base + (1 if rank < extra else 0)
    first = rank * base + min(rank, extra)
    return first, count


def expert_map_for_rank(E: int, world: int, rank: int) -> tuple[np.ndarray, int]:
    """(expert_map int32[E], local expert count) for ``rank``: owned experts map
    to 0..count-1 in order, every other expert to -1."""
    first, count = expert_partition(E, world, rank)
    emap = np.full(E, -1, np.int32)
    emap[first:first + count] = np.arange(count, dtype=np.int32)
    return emap, count


def local_weights(w: np.ndarray, E: int, world: int, rank: int) -> np.ndarray:
    """The rows of a per-expert tensor [E, ...] that ``rank`` holds."""
    first, count = expert_partition(E, world, rank)
    return w[first:first + count]


def replica_max(value: float, device=None) -> float:
    """Maximum of ``value`` over the ranks of the default process group (the
    value itself when no group is initialised).  ``device`` is where the
    one-element reduce buffer lives: a CUDA device for NCCL, the CPU for gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())

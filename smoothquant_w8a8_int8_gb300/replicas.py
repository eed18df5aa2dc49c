"""Replicas across GPUs (one process per GPU, launched by torchrun).

The linear block shards along tokens with no exchange step: every rank runs
the whole path on its own batch of tokens (weak scaling), so the only
cross-rank operations are the timing ones -- a barrier on both sides of the
timed region and the maximum of the ranks' elapsed times -- and each rank's
inputs are drawn from its own seeds.
"""
from __future__ import annotations

import os
from typing import Tuple

import torch

# Per-rank offset of every input seed.  A workload's per-GEMM seeds span less
# than a thousand values and every seed derived from one (weights, bias,
# residual, calibration and LayerNorm draws) adds at most 1,299,709, so a
# stride of 2^21 keeps the seed sets of any number of ranks disjoint.
SEED_STRIDE = 1 << 21


def rank_world() -> Tuple[int, int, int]:
    """(rank, world size, local rank) from the torchrun environment."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(seed: int, rank: int) -> int:
    """The seed of one input on `rank`: disjoint from every other rank's seeds
    (and from the seeds derived from them), reproducible per rank."""
    return seed + SEED_STRIDE * rank


def max_over_ranks(value: float, device=None) -> float:
    """The largest of the ranks' values (the job's time is its slowest rank's)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def whole_job_tops(ops_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Throughput of the whole job: the operations all ranks did per step over
    the slowest rank's step time."""
    return ops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12

"""Data-parallel replicas: one process per GPU, each serving its own batch.

The LoRA delta has no exchange between tokens, so N GPUs run N independent copies of
the hot path (weak scaling: each rank's batch has the same shape, drawn with its own
seed).  The only collectives are the ones that time the job: a barrier around the timed
region and, afterwards, the maximum of the ranks' elapsed times and the sum of the
tokens they processed.  Works with any torch.distributed backend (NCCL on GPUs, gloo on
CPU for tests).
"""
from __future__ import annotations

from typing import Tuple


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of rank ``rank``'s batch (rank 0 keeps the base seed)."""
    return int(base_seed) + int(rank)


def job_totals(elapsed_ms: float, tokens: float, device="cpu", world: int = 1) -> Tuple[float, float]:
    """(max over ranks of elapsed_ms, sum over ranks of tokens)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def tokens_per_s_per_layer(total_tokens: float, layers: int, ms_per_step: float) -> float:
    """Whole-job LoRA-delta tokens per second per layer for one step of ``ms_per_step``."""
    return total_tokens * layers / (ms_per_step / 1e3)

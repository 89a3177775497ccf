"""Whole-job throughput of independent replicas (one process per GPU).

Every (batch, head) of attention is independent, but the method is run on one
GPU per process with no sharding and no collective on the data path; several
GPUs simply run replicas of the same workload. The only cross-rank step is
the timing: the job takes as long as its slowest rank, and its throughput
is the work of all ranks divided by that time.
"""
from __future__ import annotations


def max_over_ranks(value_ms, device=None):
    """Largest value_ms over the ranks of the default process group (the
    value itself when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value_ms)
    t = torch.tensor([float(value_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flop_per_step, steps, world, max_ms):
    """TFLOP/s of `world` replicas that each ran `steps` steps of
    `flop_per_step` FLOP, the slowest in `max_ms` milliseconds."""
    if max_ms <= 0:
        raise ValueError("elapsed time must be positive")
    return world * flop_per_step * steps / (max_ms * 1e-3) / 1e12

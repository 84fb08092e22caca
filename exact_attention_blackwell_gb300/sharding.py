"""Host-side logic of the multi-GPU run: one independent copy of the workload
per rank (attention heads shard with no exchange), timing reduced with MAX.

No data-path collective exists on this path; the only collectives are the
barrier and the MAX reduction of the timed region.
"""
from __future__ import annotations


def rank_seed(seed: int, rank: int) -> int:
    """Input seed of a rank: every rank draws its own batch of the workload."""
    return seed + 1000 * rank


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's time (MAX all-reduce); identity without a process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, steps: int, max_ms: float, world: int) -> float:
    """Aggregate throughput: work of all ranks divided by the slowest rank's time."""
    return world * flops_per_rank_step * steps / (max_ms * 1e-3) / 1e12

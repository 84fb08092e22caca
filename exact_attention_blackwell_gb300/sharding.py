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


# ------------------------------------------------------------------ one problem split over ranks
# Every (batch, kv head) group is independent in both passes: the forward's
# query heads of a group read only that group's K and V, and the backward's dK
# and dV sum over the group's query heads only.  So one problem shards by
# groups with no exchange: a rank takes a contiguous block of the B * Hkv
# groups (flattened batch-major), as at most three rectangles of
# (batch range) x (kv-head range), and each rectangle is a smaller problem of
# the same shape family that the kernels solve on their own.

def group_block(B: int, Hkv: int, world: int, rank: int) -> tuple[int, int]:
    """[start, end) of this rank's groups in batch-major order; sizes differ by at most one."""
    n = B * Hkv
    return rank * n // world, (rank + 1) * n // world


def head_pieces(B: int, Hkv: int, world: int, rank: int) -> list[tuple[int, int, int, int]]:
    """This rank's groups as rectangles (b0, b1, kh0, kh1): batches b0..b1-1 x kv heads kh0..kh1-1."""
    start, end = group_block(B, Hkv, world, rank)
    if start >= end:
        return []
    bs, khs = divmod(start, Hkv)
    be, khe = divmod(end, Hkv)  # end is exclusive
    if bs == be:
        return [(bs, bs + 1, khs, khe)]
    pieces = []
    if khs > 0:  # a partial first batch
        pieces.append((bs, bs + 1, khs, Hkv))
        bs += 1
    if be > bs:  # whole batches
        pieces.append((bs, be, 0, Hkv))
    if khe > 0:  # a partial last batch
        pieces.append((be, be + 1, 0, khe))
    return pieces


def slice_piece(t, piece, heads_per_group: int = 1, head_dim: int = 2):
    """The piece's part of a tensor whose head axis is `head_dim` (2 for [B, N, heads, d],
    1 for [B, heads, N]); query-head tensors pass the group size H / Hkv."""
    b0, b1, kh0, kh1 = piece
    idx = [slice(None)] * t.dim()
    idx[0] = slice(b0, b1)
    idx[head_dim] = slice(kh0 * heads_per_group, kh1 * heads_per_group)
    return t[tuple(idx)].contiguous()

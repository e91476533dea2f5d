"""Sequence sharding across GPUs (one process per GPU).

Verification of one sequence never reads another sequence's data, so a batch
splits across ranks by sequence with no collective on the data path.  The
Philox counter is keyed on the global sequence index (``seq_offset + b``), so
a sharded batch draws exactly the uniforms the whole batch would.
"""
from __future__ import annotations


def shard_bounds(B: int, world_size: int, rank: int) -> tuple[int, int]:
    """[lo, hi) of the sequences rank `rank` verifies out of a batch of B
    (contiguous blocks; the first B % world_size ranks get one extra)."""
    if world_size < 1 or not 0 <= rank < world_size or B < 0:
        raise ValueError(f"bad shard request B={B} world_size={world_size} rank={rank}")
    base, extra = divmod(B, world_size)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def weak_scaling_offset(B_per_rank: int, rank: int) -> int:
    """seq_offset of a rank that verifies its own batch of B_per_rank sequences
    (weak scaling): global sequence ids rank * B_per_rank + b."""
    return rank * B_per_rank

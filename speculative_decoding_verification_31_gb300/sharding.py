"""Batch sharding over GPUs: contiguous ranges of sequences with their global index.

The verify step is independent per sequence and its random numbers are keyed by the global
sequence index, so a batch split over N GPUs (each calling the library on its own range
with ``seq_index_base`` = the range's first global index) gives exactly the tokens one GPU
would give for the whole batch.  No collective is needed on the data path.
"""
from __future__ import annotations


def shard_range(total: int, world: int, rank: int) -> tuple[int, int]:
    """[lo, hi) of the sequences owned by `rank` of `world`: contiguous, sizes differing by
    at most one, the first `total % world` ranks taking the extra sequence."""
    if world < 1 or not 0 <= rank < world or total < 0:
        raise ValueError(f"bad shard request: total={total} world={world} rank={rank}")
    base, extra = divmod(total, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi

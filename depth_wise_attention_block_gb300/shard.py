"""Token sharding across ranks.

Every token's depth aggregation is independent of every other token's
(the sources, weights and output of token t are row t of their tensors), so
a batch splits across GPUs by contiguous token ranges with no exchange of
data: each rank holds the rows of its tokens of h_0, the block sums and the
partial sum, and a copy of the 28 KB pseudo-queries.
"""
from __future__ import annotations


def token_range(T: int, rank: int, world: int) -> tuple[int, int]:
    """[start, end) of the tokens rank `rank` of `world` owns: contiguous,
    sizes differing by at most one, in rank order, covering [0, T)."""
    if world < 1 or not (0 <= rank < world) or T < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, T >= 0")
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)

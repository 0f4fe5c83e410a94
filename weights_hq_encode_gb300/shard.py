"""Splitting one tensor's tiles across ranks (GPUs) with no data-path exchange.

The codec is data-parallel over tiles (every tile codes independently given
its global index, which keys the dither).  A rank codes a contiguous,
group-aligned range of tiles with ``tile_base`` = the range's first tile, so
its stream is exactly the corresponding slice of the stream one call over the
whole tensor would produce (groups start on word boundaries).  Turning the
per-rank streams into one global stream needs one exchange only: an
exclusive scan of the per-rank word totals, which shifts each rank's index.
"""
from __future__ import annotations

GROUP_TILES = 32


def shard_range(n_tiles: int, world: int, rank: int) -> tuple[int, int]:
    """[begin, end) tiles of `rank`: group-aligned, balanced to within a group."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    n_groups = (n_tiles + GROUP_TILES - 1) // GROUP_TILES
    g0 = (n_groups * rank) // world
    g1 = (n_groups * (rank + 1)) // world
    return min(g0 * GROUP_TILES, n_tiles), min(g1 * GROUP_TILES, n_tiles)


def merge_offsets(per_rank_offsets):
    """Global index from per-rank indices (each: n_groups_r + 1 word offsets
    starting at 0): rank r's entries are shifted by the words of ranks < r;
    the shared boundary entries coincide."""
    merged, base = [], 0
    for r, off in enumerate(per_rank_offsets):
        off = [int(v) for v in off]
        if off and off[0] != 0:
            raise ValueError("per-rank index must start at 0")
        body = off[:-1] if r < len(per_rank_offsets) - 1 else off
        merged.extend(base + v for v in body)
        base += off[-1] if off else 0
    return merged


def exclusive_word_base(totals, rank: int) -> int:
    """Word offset of `rank`'s stream in the global stream."""
    return sum(int(t) for t in totals[:rank])

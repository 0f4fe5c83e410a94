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


class RankCode:
    """One rank's part of a sharded encode: its tile range, its stream and
    index (local, starting at word 0), and where they sit in the global
    stream."""

    def __init__(self, begin, end, stream, offsets, total_words, status, word_base, totals):
        self.begin, self.end = begin, end
        self.stream, self.offsets = stream, offsets
        self.total_words, self.status = total_words, status
        self.word_base, self.totals = word_base, totals

    def global_offsets(self):
        """This rank's index entries shifted into the global stream (the last
        entry is the next rank's first)."""
        return [self.word_base + int(v) for v in self.offsets]


def code_rank(n_tiles: int, world: int, rank: int, encode_range, allgather_int) -> RankCode:
    """Sharded encode of one tensor of `n_tiles` tiles: this rank codes its
    group-aligned range [b, e) with `encode_range(b, e)` (which must use
    tile_base = b, so that the dither counters are the global tile indices)
    -> (stream, offsets starting at 0, total_words, status); the one exchange,
    `allgather_int(total_words)` -> every rank's total, gives the rank's word
    offset in the global stream.  The concatenation of the ranks' streams in
    rank order is, word for word, the stream of one call over the whole
    tensor, and merge_offsets of their indices its index."""
    b, e = shard_range(n_tiles, world, rank)
    stream, offsets, total, status = encode_range(b, e)
    totals = [int(t) for t in allgather_int(int(total))]
    if len(totals) != world or totals[rank] != int(total):
        raise RuntimeError("inconsistent word totals from the all-gather")
    return RankCode(b, e, stream, offsets, int(total), int(status),
                    exclusive_word_base(totals, rank), totals)


def device_encode_range(hq, params, x_tiles, x_first: int = 0):
    """encode_range for code_rank on this rank's GPU: hq_encode (size query,
    then the encode) over global tiles [b, e), held by `x_tiles` (a CUDA int16
    view [n, 128] of bf16 data whose row 0 is global tile `x_first`), with
    `params` copied and its tile_base set to b."""
    import torch

    def run(b, e):
        n = e - b
        dev = x_tiles.device
        p = type(params).from_buffer_copy(params)     # a copy of the C struct's bytes
        for keep in ("_signs", "_rot"):                # the device arrays it points to
            if hasattr(params, keep):
                setattr(p, keep, getattr(params, keep))
        p.tile_base = b
        if b < x_first or e - x_first > x_tiles.shape[0]:
            raise ValueError("the rank's tile range is not held by x_tiles")
        xs = x_tiles[b - x_first:e - x_first]
        offsets = torch.zeros(hq.hq_num_groups(n) + 1, dtype=torch.int64, device=dev)
        ws = torch.zeros(max(hq.hq_encode_workspace_bytes(n), 8), dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if hq.hq_encode(p, xs, n, None, 0, offsets, ws, status) != hq.HQ_OK:
            raise RuntimeError("hq_encode (size query) failed")
        total = int(offsets[-1].item()) if n > 0 else 0
        stream = torch.empty(max(total, 1), dtype=torch.int32, device=dev)
        status.zero_()
        if hq.hq_encode(p, xs, n, stream, total, offsets, ws, status) != hq.HQ_OK:
            raise RuntimeError("hq_encode failed")
        return stream, offsets.cpu().numpy().view("uint64").tolist(), total, int(status.item())

    return run

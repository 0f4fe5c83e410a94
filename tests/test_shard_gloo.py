"""Multi-rank path on CPU (gloo, world size 2): shard.code_rank -- the rank
function bench.py runs on GPUs -- codes each rank's group-aligned tile range
with tile_base = its first tile; the per-rank streams, joined through one
all-gather of word totals, equal the stream of one call over the whole
tensor, bit for bit.  Only the device call is replaced: the CPU oracle codes
the range here, hq_encode on the rank's GPU in bench.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        from oracle import oracle as O
        from weights_hq_encode_gb300 import inputs as I, shard
        x = I.bf16_bits(I.tiny_kv()).reshape(-1, 128)
        x = np.concatenate([x, x[:77]])                     # 333 tiles: ragged last group
        def encode_range(b, e):                            # the oracle stands in for hq_encode
            P = O.make_params(8, 2, 1.7, 1, 7, O.make_signs(0, 0), 1 << 40, tile_base=b)
            enc = O.encode(P, x[b:e], threads=1)
            return enc["stream"], enc["offsets"].tolist(), enc["total_words"], enc["status"]

        def allgather_int(v):                              # the one exchange
            totals = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(totals, torch.tensor([v], dtype=torch.int64))
            return [int(t.item()) for t in totals]

        rc = shard.code_rank(x.shape[0], world, rank, encode_range, allgather_int)
        assert rc.status == 0
        # gather streams and indices (test only: a deployment keeps them sharded)
        objs = [None] * world
        dist.all_gather_object(objs, (rc.word_base, rc.stream.tolist(), rc.offsets,
                                      rc.global_offsets()))
        if rank == 0:
            stream = [w for _, s, _, _ in sorted(objs, key=lambda o: o[0]) for w in s]
            offsets = shard.merge_offsets([o for _, _, o, _ in objs])
            glob = [v for _, _, _, g in objs[:-1] for v in g[:-1]] + objs[-1][3]
            assert glob == offsets
            np.savez(result_path, stream=np.array(stream, np.uint64), offsets=np.array(offsets, np.uint64))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reproduce_the_single_call_stream(tmp_path, oracle):
    world, port = 2, _free_port()
    res = str(tmp_path / "merged.npz")
    mp.start_processes(_rank_main, args=(world, port, res), nprocs=world, start_method="spawn",
                       join=True)
    got = np.load(res)
    from weights_hq_encode_gb300 import inputs as I
    x = I.bf16_bits(I.tiny_kv()).reshape(-1, 128)
    x = np.concatenate([x, x[:77]])
    P = oracle.make_params(8, 2, 1.7, 1, 7, oracle.make_signs(0, 0), 1 << 40)
    ref = oracle.encode(P, x)
    assert (got["offsets"] == ref["offsets"]).all()
    assert (got["stream"].astype(np.uint32) == ref["stream"]).all()


def test_shard_ranges_cover_and_align():
    from weights_hq_encode_gb300 import shard
    for n in (0, 1, 31, 32, 33, 1000, 4194304):
        for world in (1, 2, 3, 8):
            rs = [shard.shard_range(n, world, r) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == n
            for (b0, e0), (b1, e1) in zip(rs, rs[1:]):
                assert e0 == b1 and b1 % 32 == 0
    assert shard.merge_offsets([[0, 3, 5], [0, 2]]) == [0, 3, 5, 7]

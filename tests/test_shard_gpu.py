"""The sharded encode on the GPU: shard.code_rank with device_encode_range
(hq_encode on this device over a rank's group-aligned tile range, tile_base
= its first tile) for 2 and 3 ranks run one after another in this process,
the all-gather of word totals replaced by the totals the ranks report.  The
ranks' streams, concatenated in rank order, and their merged indices must
equal the oracle's single encode of the whole tensor, bit for bit."""
import numpy as np
import pytest
import torch

from _cases import bits_to_torch, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq as H
    return H


@pytest.mark.parametrize("world,local", [(2, False), (3, False), (3, True)])
def test_code_rank_on_the_gpu_reproduces_the_single_call(hq, oracle, world, local):
    from weights_hq_encode_gb300 import shard
    rng = np.random.default_rng(40 + world)
    n = 1000                                               # ragged last group
    xf = rng.standard_normal((n, 128)).astype(np.float32)
    xb = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    x = bits_to_torch(xb)
    mask = oracle.make_signs(9, 0).reshape(1, 4)
    signs = torch.from_numpy(mask.view(np.int32).copy()).cuda()
    p = hq.make_params(hq.HQ_E8, 2, 1.9, 1, 77, signs, 1 << 40)

    def encode_range_for(rank):
        if not local:
            return shard.device_encode_range(hq, p, x)
        b, e = shard.shard_range(n, world, rank)          # the rank holds only its tiles
        return shard.device_encode_range(hq, p, x[b:e].clone(), x_first=b)

    totals = [encode_range_for(r)(*shard.shard_range(n, world, r))[2] for r in range(world)]
    ranks = [shard.code_rank(n, world, r, encode_range_for(r), lambda v: totals)
             for r in range(world)]
    assert all(rc.status == 0 for rc in ranks)
    stream = np.concatenate([u32(rc.stream[:rc.total_words]) for rc in ranks])
    offsets = shard.merge_offsets([rc.offsets for rc in ranks])
    glob = [v for rc in ranks[:-1] for v in rc.global_offsets()[:-1]] + ranks[-1].global_offsets()
    assert glob == offsets
    ref = oracle.encode(oracle.make_params(8, 2, 1.9, 1, 77, mask, 1 << 40), xb)
    assert (np.array(offsets, np.uint64) == ref["offsets"]).all()
    assert (stream == ref["stream"]).all()
    assert [rc.word_base for rc in ranks] == [sum(totals[:r]) for r in range(world)]

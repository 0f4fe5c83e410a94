"""hq_encode_noalloc: the encoder for callers that cannot allocate device
memory (a serving engine whose allocator owns all free memory, a path where
cudaMalloc's device synchronisation is not allowed, a plugin given no
allocator).  It uses the library's built-in scratch instead of a caller
workspace; its output must equal hq_encode's, call after call, because every
call clears the shared scratch it inherits from the previous one.

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq as H
    return H


def p_signs(hq, seed):
    m = hq.hq_make_layer_signs(seed, seed + 1, 0)
    return torch.from_numpy(np.asarray(m, np.uint32).view(np.int32).reshape(1, 4)).cuda()


def _inputs(hq, n, seed, k, alpha):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((n, 128)).astype(np.float32)).to(torch.bfloat16)
    x = x.cuda().view(torch.int16)
    return x, hq.make_params(hq.HQ_E8, k, alpha, 1, seed, p_signs(hq, seed), 1 << 40)


def _with_workspace(hq, p, x, n):
    offsets = torch.zeros(hq.hq_num_groups(n) + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(hq.hq_encode_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_encode(p, x, n, None, 0, offsets, ws, status) == hq.HQ_OK
    total = int(offsets[-1].item())
    stream = torch.empty(total, dtype=torch.int32, device="cuda")
    status.zero_()
    assert hq.hq_encode(p, x, n, stream, total, offsets, ws, status) == hq.HQ_OK
    torch.cuda.synchronize()
    return stream.cpu(), offsets.cpu(), int(status.item()), total


def test_noalloc_matches_hq_encode_on_consecutive_calls(hq):
    # two different inputs in a row: the second call inherits the first call's scratch
    for n, seed, k, alpha in ((3000, 11, 2, 1.7), (777, 12, 1, 0.6), (3000, 11, 2, 1.7)):
        x, p = _inputs(hq, n, seed, k, alpha)
        ref_stream, ref_offsets, ref_status, total = _with_workspace(hq, p, x, n)
        offsets = torch.full((hq.hq_num_groups(n) + 1,), -1, dtype=torch.int64, device="cuda")
        stream = torch.full((total + 4,), -1, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert hq.hq_encode_noalloc(p, x, n, stream, total, offsets, status) == hq.HQ_OK
        torch.cuda.synchronize()
        assert int(status.item()) == ref_status == 0
        assert torch.equal(offsets.cpu(), ref_offsets)
        assert torch.equal(stream[:total].cpu(), ref_stream)
        assert (stream[total:].cpu() == -1).all()


def test_noalloc_allocates_nothing_and_covers_its_other_modes(hq):
    """After a first call (which looks up the scratch address), further calls
    leave the device's free memory unchanged; the size-query mode (no output
    buffer) gives hq_encode's index; a params block carrying
    HQ_FLAG_WORKSPACE_READY codes identically (the flag is ignored: the shared
    scratch is always cleared)."""
    n = 1500
    x, p = _inputs(hq, n, 21, 2, 1.3)
    ref_stream, ref_offsets, ref_status, total = _with_workspace(hq, p, x, n)
    offsets = torch.zeros(hq.hq_num_groups(n) + 1, dtype=torch.int64, device="cuda")
    stream = torch.full((total + 4,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_encode_noalloc(p, x, n, stream, total, offsets, status) == hq.HQ_OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(4):
        assert hq.hq_encode_noalloc(p, x, n, stream, total, offsets, status) == hq.HQ_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    # size query: only the index and the status are written, as by hq_encode
    # (which flags HQ_ERR_CAPACITY there: the zero capacity is below the need)
    ws = torch.empty(hq.hq_encode_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    ref_q = torch.zeros(hq.hq_num_groups(n) + 1, dtype=torch.int64, device="cuda")
    ref_st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_encode(p, x, n, None, 0, ref_q, ws, ref_st) == hq.HQ_OK
    offsets.fill_(-1)
    status.zero_()
    assert hq.hq_encode_noalloc(p, x, n, None, 0, offsets, status) == hq.HQ_OK
    torch.cuda.synchronize()
    assert torch.equal(offsets.cpu(), ref_offsets) and torch.equal(ref_q.cpu(), ref_offsets)
    assert int(status.item()) == int(ref_st.item())
    status.zero_()
    # a caller's "workspace ready" flag changes nothing
    pf = hq.make_params(hq.HQ_E8, 2, 1.3, 1, 21, p_signs(hq, 21), 1 << 40,
                        flags=hq.HQ_FLAG_WORKSPACE_READY)
    stream.fill_(-1)
    offsets.fill_(-1)
    assert hq.hq_encode_noalloc(pf, x, n, stream, total, offsets, status) == hq.HQ_OK
    torch.cuda.synchronize()
    assert int(status.item()) == ref_status == 0
    assert torch.equal(offsets.cpu(), ref_offsets)
    assert torch.equal(stream[:total].cpu(), ref_stream)


def test_noalloc_rejects_more_tiles_than_its_scratch(hq):
    x, p = _inputs(hq, 1, 13, 2, 1.0)
    offsets = torch.zeros(2, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hq.hq_encode_noalloc(p, x, hq.HQ_NOALLOC_MAX_TILES + 1, None, 0, offsets, status)
    assert rc == hq.HQ_ERR_INVALID

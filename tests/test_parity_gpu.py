"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Codes, bitstreams and group indices must be bit-identical; decoded fp32 must
be within 1e-5 relative (per tile, l2) and is expected bit-identical; bf16
output must be bit-identical.  Sizes span several blocks of 128 tiles and
ragged tails; the full-size workloads (KV cache, weight matrices, the
long-context sweep, the fused-scores keys) are compared whole: every stream
word, every index entry and every bf16 decoded value."""
import numpy as np
import pytest
import torch

from _cases import Case, bits_to_torch, calibration, gpu_decode, gpu_encode, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq as H
    return H


def _rel_l2_per_tile(a, b):
    num = np.sqrt(((a.astype(np.float64) - b) ** 2).sum(-1))
    den = np.sqrt((b.astype(np.float64) ** 2).sum(-1)) + 1e-30
    return num / den


def _check_case(hq, O, c: Case, check_decode=True):
    P = c.oracle_params(O)
    ref = O.encode(P, c.x_bits)
    x = bits_to_torch(c.x_bits)
    p = c.gpu_params(hq)
    stream, offsets, status, total, _ = gpu_encode(hq, p, x, c.n)
    assert status == ref["status"]
    assert (offsets.cpu().numpy().view(np.uint64) == ref["offsets"]).all()
    assert total == ref["total_words"]
    s = u32(stream)
    assert (s[:total] == ref["stream"][:total]).all()
    assert (s[total:] == 0xFFFFFFFF).all()                  # nothing written past the end
    if not check_decode:
        return stream, offsets, total
    dref = O.decode(P, ref["stream"], ref["offsets"], c.n)
    dref_b = O.decode(P, ref["stream"], ref["offsets"], c.n, out="bf16")
    out, st = gpu_decode(hq, p, stream, total, offsets, c.n, hq.HQ_OUT_F32)
    assert st == dref["status"] == 0
    o = out.cpu().numpy()
    assert np.all(_rel_l2_per_tile(o, dref["out"]) <= 1e-5)
    assert (o.view(np.uint32) == dref["out"].view(np.uint32)).mean() == 1.0
    outb, st = gpu_decode(hq, p, stream, total, offsets, c.n, hq.HQ_OUT_BF16)
    assert st == 0
    assert (outb.cpu().view(torch.int16).numpy().view(np.uint16) == dref_b["out"]).all()
    return stream, offsets, total


def _rand_bits(rng, n, scale=1.0, outliers=0.01):
    x = rng.standard_normal((n, 128)).astype(np.float32) * scale
    hit = rng.random((n, 128)) < outliers
    x[hit] *= 20
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


CASES = [
    # lattice, k, alpha, dither, n_tiles, n_segments, tile_base
    (8, 2, 1.7, 1, 256, 1, 0),
    (8, 0, 1.0, 1, 1, 1, 0),
    (8, 1, 0.4, 1, 17, 2, 5),
    (8, 3, 4.0, 0, 33, 3, 0),
    (8, 2, 2.5, 1, 129, 4, 123456789),
    (8, 5, 40.0, 1, 300, 1, 0),
    (8, 1, 0.05, 1, 70, 1, 0),
    (8, 0, 300.0, 1, 40, 1, 0),       # groups far beyond the encoder's shared staging
    (8, 2, 60.0, 0, 520, 2, 3),       # several blocks of 4 groups, ragged tail
    (4, 0, 0.8, 1, 65, 2, 0),
    (4, 1, 1.3, 1, 200, 1, 7),
    (4, 3, 6.0, 0, 31, 1, 0),
    (2, 0, 0.9, 1, 90, 1, 0),         # A2 (hexagonal), parity copies written at k = 0
    (2, 1, 1.5, 1, 260, 2, 11),
    (2, 3, 5.0, 0, 47, 1, 0),
    (2, 6, 120.0, 1, 33, 1, 0),       # generic-width remainders
    (1, 0, 0.3, 1, 100, 1, 0),
    (1, 2, 2.0, 1, 257, 3, 99),
    (1, 4, 16.0, 0, 64, 1, 0),
]


@pytest.mark.parametrize("lat,k,alpha,dither,n,nseg,base", CASES)
def test_small_cases_bit_exact(hq, oracle, lat, k, alpha, dither, n, nseg, base):
    rng = np.random.default_rng(1000 + n + k)
    x = _rand_bits(rng, n)
    masks = np.stack([oracle.make_signs(77, s) for s in range(nseg)])
    tps = max(1, -(-n // nseg))
    _check_case(hq, oracle, Case(x, lat, k, alpha, dither, 4242 + n, masks, tps, base))


@pytest.mark.parametrize("lat,k,alpha,dither,n,nseg", [
    (8, 2, 1.7, 1, 160, 2),        # Haar rotation per segment (32-tile aligned segments)
    (8, 0, 0.6, 1, 70, 1),
    (4, 1, 1.3, 0, 96, 3),
    (2, 2, 2.0, 1, 64, 2),
    (1, 3, 6.0, 1, 33, 1),
])
def test_dense_rotation_bit_exact(hq, oracle, lat, k, alpha, dither, n, nseg):
    """The per-layer Haar (QJL) rotation: codes, streams and decodes equal the
    oracle's fixed-order fp32 chains bit for bit."""
    from weights_hq_encode_gb300 import inputs as I
    rng = np.random.default_rng(2000 + n + k)
    x = _rand_bits(rng, n)
    masks = np.stack([oracle.make_signs(78, s) for s in range(nseg)])
    tps = 32 * max(1, -(-n // (32 * nseg)))
    rot = I.haar_rotations(nseg, seed=500 + n)
    _check_case(hq, oracle, Case(x, lat, k, alpha, dither, 77 + n, masks, tps, 0, rot=rot))


def test_dense_rotation_needs_aligned_segments(hq, oracle):
    from weights_hq_encode_gb300 import inputs as I
    x = torch.zeros((40, 128), dtype=torch.int16, device="cuda")
    c = Case(np.zeros((40, 128), np.uint16), 8, 2, 1.0, 1, 1, oracle.make_signs(1, 0), 20,
             rot=I.haar_rotations(2))
    p = c.gpu_params(hq)
    offsets = torch.zeros(hq.hq_num_groups(40) + 1, dtype=torch.int64, device="cuda")
    ws = torch.zeros(hq.hq_encode_workspace_bytes(40), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_encode(p, x, 40, None, 0, offsets, ws, st) == hq.HQ_ERR_INVALID


def test_tiny_kv_config(hq, oracle):
    from weights_hq_encode_gb300 import inputs as I
    cal = calibration()["tiny_kv"]["E8"]["3.0"]
    x = I.bf16_bits(I.tiny_kv())
    c = Case(x, 8, cal["k"], cal["alpha"], 1, I.TINY["dither_seed"],
             oracle.make_signs(I.TINY["sign_seed"], 0), 1 << 40)
    _check_case(hq, oracle, c)


def test_empty_and_special_inputs(hq, oracle):
    # zero tiles, constant tiles, huge and non-finite tiles (range rule), bf16 subnormals
    x = np.zeros((40, 128), np.uint16)
    x[1] = 0x3F80                                           # all ones
    x[2, ::2] = 0x8000                                      # -0
    x[3, 7] = 0x7F7F                                        # max finite bf16
    x[4, 9] = 0x7F80                                        # +inf
    x[5, 0] = 0x7FC1                                        # NaN
    x[6] = 0x0001                                           # subnormal
    x[7, 3] = 0x4B00                                        # 2^23
    for lat in (8, 4, 1):
        c = Case(x, lat, 2, 3.0, 1, 5, oracle.make_signs(1, 0), 1 << 40)
        _check_case(hq, oracle, c)
    # n_tiles = 0: only offsets[0] = 0 is written
    p = Case(x[:0], 8, 2, 3.0, 1, 5, oracle.make_signs(1, 0), 1 << 40).gpu_params(hq)
    offsets = torch.full((1,), 99, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(8, dtype=torch.uint8, device="cuda")
    assert hq.hq_encode(p, bits_to_torch(x), 0, None, 0, offsets, ws, status) == hq.HQ_OK
    torch.cuda.synchronize()
    assert int(offsets[0]) == 0 and int(status[0]) == 0


def test_capacity(hq, oracle):
    rng = np.random.default_rng(3)
    x = _rand_bits(rng, 1000)
    c = Case(x, 8, 2, 2.0, 1, 9, oracle.make_signs(3, 0), 1 << 40)
    P = c.oracle_params(oracle)
    full = oracle.encode(P, x)
    cap = full["total_words"] // 3
    part = oracle.encode(P, x, cap_words=cap)
    stream, offsets, status, total, _ = gpu_encode(hq, c.gpu_params(hq), bits_to_torch(x), c.n,
                                                   cap=cap)
    assert status == part["status"] and status & hq.HQ_ERR_CAPACITY
    assert (offsets.cpu().numpy().view(np.uint64) == full["offsets"]).all()
    s = u32(stream)
    assert (s[:cap] == full["stream"][:cap]).all() and (s[cap:] == 0xFFFFFFFF).all()


def test_corrupt_streams(hq, oracle):
    rng = np.random.default_rng(4)
    x = _rand_bits(rng, 200)
    c = Case(x, 8, 1, 0.6, 1, 10, oracle.make_signs(4, 0), 1 << 40)
    P = c.oracle_params(oracle)
    ref = oracle.encode(P, x)
    p = c.gpu_params(hq)
    for trial in range(12):
        s = ref["stream"].copy()
        off = ref["offsets"].copy()
        if trial < 8:
            w = int(rng.integers(0, s.size))
            s[w] ^= np.uint32(1 << int(rng.integers(0, 32)))
        elif trial < 10:
            off[int(rng.integers(1, off.size))] += np.uint64(1)
        elif trial == 10:
            off[3] = np.uint64(10 ** 12)                    # index points far outside the stream
        else:
            s[:] = 0
        d = oracle.decode(P, s, off, c.n)
        out, st = gpu_decode(hq, p, bits_to_torch(s.view(np.uint16)).view(torch.int32),
                             int(s.size), bits_to_torch(off.view(np.uint16)).view(torch.int64),
                             c.n, hq.HQ_OUT_F32)
        assert st == d["status"]
        o = out.cpu().numpy()
        assert (o.view(np.uint32) == d["out"].view(np.uint32)).all()


def test_lookback_timeout_is_reported(hq, oracle):
    """A predecessor flag that nothing sets (ticket counter pre-set to 1):
    the bounded wait runs out and the encoder reports HQ_ERR_TIMEOUT."""
    rng = np.random.default_rng(5)
    x = _rand_bits(rng, 1024)
    c = Case(x, 8, 2, 2.0, 1, 11, oracle.make_signs(5, 0), 1 << 40)
    p = c.gpu_params(hq, lookback_spins=2000, flags=hq.HQ_FLAG_WORKSPACE_READY)
    n = c.n
    xt = bits_to_torch(x)
    offsets = torch.zeros(hq.hq_num_groups(n) + 1, dtype=torch.int64, device="cuda")
    ws = torch.zeros(hq.hq_encode_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    ws[0] = 1                                               # ticket counter starts at 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    assert hq.hq_encode(p, xt, n, stream, 1 << 16, offsets, ws, status) == hq.HQ_OK
    torch.cuda.synchronize()
    assert int(status.item()) & hq.HQ_ERR_TIMEOUT
    # the context is still usable: a normal encode right after is bit-exact
    _check_case(hq, oracle, c, check_decode=False)


def test_prepared_workspace_codes_identically(hq, oracle):
    """With HQ_FLAG_WORKSPACE_READY the library skips its workspace memset and
    the blocks take their groups from the caller-zeroed ticket counter: the
    stream, index and status are the same bit for bit."""
    rng = np.random.default_rng(6)
    x = _rand_bits(rng, 777)
    c = Case(x, 8, 2, 2.0, 1, 12, oracle.make_signs(6, 0), 1 << 40)
    ref = oracle.encode(c.oracle_params(oracle), c.x_bits)
    p = c.gpu_params(hq, flags=hq.HQ_FLAG_WORKSPACE_READY)
    xt = bits_to_torch(x)
    offsets = torch.zeros(hq.hq_num_groups(c.n) + 1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.full((ref["total_words"] + 8,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):                                  # the caller re-zeroes between calls
        ws = torch.zeros(hq.hq_encode_workspace_bytes(c.n), dtype=torch.uint8, device="cuda")
        assert hq.hq_encode(p, xt, c.n, stream, ref["total_words"], offsets, ws, status) == hq.HQ_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert (offsets.cpu().numpy().view(np.uint64) == ref["offsets"]).all()
        assert (u32(stream)[:ref["total_words"]] == ref["stream"][:ref["total_words"]]).all()


def test_invalid_arguments(hq, oracle):
    x = bits_to_torch(np.zeros((4, 128), np.uint16))
    c = Case(np.zeros((4, 128), np.uint16), 8, 2, 1.0, 1, 0, oracle.make_signs(0, 0), 1 << 40)
    offsets = torch.zeros(2, dtype=torch.int64, device="cuda")
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (dict(lattice=3), dict(rice_k=16), dict(alpha=0.0), dict(alpha=float("nan")),
                dict(dither=2), dict(tiles_per_segment=0)):
        p = c.gpu_params(hq)
        for kk, vv in bad.items():
            setattr(p, kk, vv)
        assert hq.hq_encode(p, x, 4, None, 0, offsets, ws, status) == hq.HQ_ERR_INVALID
    p = c.gpu_params(hq)
    big = torch.zeros(5 * 128, dtype=torch.int16, device="cuda")
    xm = big[1:1 + 4 * 128]                                  # 2-byte offset: misaligned input
    assert xm.data_ptr() % 16 == 2
    assert hq.hq_encode(p, xm, 4, None, 0, offsets, ws, status) == hq.HQ_ERR_INVALID
    small_ws = torch.zeros(8, dtype=torch.uint8, device="cuda")
    assert hq.hq_encode(p, x, 4, None, 0, offsets, small_ws, status) == hq.HQ_ERR_INVALID


# ---------------------------------------------------------------- full-size workloads
def _whole(hq, oracle, xt, n, P, p, decode=True):
    """Encode the whole workload on both sides and compare every word of the
    stream, every index entry and the status; then decode the whole stream to
    bf16 on both sides and compare every value.  Returns (stream, offsets,
    total) of the GPU encode."""
    xb = xt.cpu().numpy().view(np.uint16).reshape(-1, 128)
    ref = oracle.encode(P, xb)
    stream, offsets, status, total, _ = gpu_encode(hq, p, xt, n)
    assert status == ref["status"] == 0
    assert total == ref["total_words"]
    assert (offsets.cpu().numpy().view(np.uint64) == ref["offsets"]).all()
    s = u32(stream)
    assert (s[:total] == ref["stream"][:total]).all()
    assert (s[total:] == 0xFFFFFFFF).all()
    del xb, s
    if decode:
        out, st = gpu_decode(hq, p, stream, total, offsets, n, hq.HQ_OUT_BF16)
        assert st == 0
        got = out.cpu().view(torch.int16).numpy().view(np.uint16)
        del out
        dref = oracle.decode(P, ref["stream"], ref["offsets"], n, out="bf16")
        assert dref["status"] == 0
        assert np.array_equal(got, dref["out"])
    return stream, offsets, total


@pytest.mark.parametrize("rate", ["2.0", "3.0"])
def test_kv_cache_8b_whole(hq, oracle, rate):
    """The Llama-3.1-8B-shaped KV cache (32 layers x K,V x 8 heads x 8192
    tokens, per-layer sign rotation, dither, E8): the whole stream, index and
    bf16 decode equal the oracle's; the realized rate is within 0.01 bps."""
    from weights_hq_encode_gb300 import inputs as I
    C = I.KV8B
    cal = calibration()["kv_cache_8b"]["E8"][rate]
    x = I.kv_cache_8b("cuda")
    n = x.numel() // 128
    masks = hq.kv_layer_masks(C["sign_seed"], C["layer_sign_seed"], C["layers"])
    seg = np.array([masks[l] for l in range(C["layers"]) for _ in (0, 1)], np.uint32)
    tps = C["kv_heads"] * C["tokens"]
    signs = torch.from_numpy(seg.view(np.int32).copy()).cuda()
    p = hq.make_params(8, cal["k"], cal["alpha"], 1, C["dither_seed"], signs, tps)
    P = oracle.make_params(8, cal["k"], cal["alpha"], 1, C["dither_seed"], seg, tps)
    xt = hq.as_tiles(x)
    del x
    stream, offsets, total = _whole(hq, oracle, xt, n, P, p)
    bps = (total * 32 - 15.5 * hq.hq_num_groups(n)) / (n * 128)
    assert abs(bps - float(rate)) < 0.01, bps
    # fp32 decode of sampled groups is within 1e-5 (and in practice equal to) the oracle's
    outf, st = gpu_decode(hq, p, stream, total, offsets, n, hq.HQ_OUT_F32)
    assert st == 0
    rng = np.random.default_rng(int(float(rate) * 10))
    for g in [0, hq.hq_num_groups(n) - 1] + rng.integers(0, hq.hq_num_groups(n), 6).tolist():
        t0 = 32 * g
        xb = xt[t0:t0 + 32].cpu().numpy().view(np.uint16)
        Pg = oracle.make_params(8, cal["k"], cal["alpha"], 1, C["dither_seed"],
                                seg[t0 // tps].reshape(1, 4), 1 << 40, t0)
        ref = oracle.encode(Pg, xb)
        d = oracle.decode(Pg, ref["stream"], ref["offsets"], xb.shape[0])
        assert np.all(_rel_l2_per_tile(outf[t0:t0 + 32].cpu().numpy(), d["out"]) <= 1e-5)


@pytest.mark.parametrize("rate", ["2.0", "3.0"])
def test_kv_cache_8b_e8_rule_census(oracle, rate):
    """On the KV-cache inputs, how often the codec's E8 coset test (an fp32
    evaluation of the exact linear identity for the difference of the two
    squared distances) and the plain rule (the two fp32 squared distances
    summed left to right) pick different points: only at exact-distance
    near-ties, and rarely.  The inputs are the GPU-drawn cache, read back."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import inputs as I
    from weights_hq_encode_gb300 import hq
    C = I.KV8B
    cal = calibration()["kv_cache_8b"]["E8"][rate]
    x = I.kv_cache_8b("cuda")
    xb = x.reshape(-1, 128).view(torch.int16).cpu().numpy().view(np.uint16)
    del x
    masks = hq.kv_layer_masks(C["sign_seed"], C["layer_sign_seed"], C["layers"])
    seg = np.array([masks[l] for l in range(C["layers"]) for _ in (0, 1)], np.uint32)
    P = oracle.make_params(8, cal["k"], cal["alpha"], 1, C["dither_seed"], seg,
                           C["kv_heads"] * C["tokens"])
    c = oracle.e8_rule_census(P, xb)
    print(f"\nE8 rule census, KV cache at {rate} bps: {c}")
    assert c["vectors"] == xb.shape[0] * 16
    assert c["differ"] <= 1e-6 * c["vectors"]
    assert c["dist_max"] <= 1e-3
    # the same inputs: scale and dither rounded once (the codec) or twice
    r = oracle.scale_rounding_census(P, xb)
    print(f"scale rounding census, KV cache at {rate} bps: {r}")
    assert r["vectors"] == xb.shape[0] * 16 and r["skipped_tiles"] == 0
    assert r["differ"] <= 1e-5 * r["vectors"]


@pytest.mark.parametrize("rate", ["3.0", "4.0", "5.0"])
def test_weights_8b_whole(hq, oracle, rate):
    """The four Llama-3.1-8B linear-weight shapes at 3, 4 and 5 bps (no
    dither, one sign mask): whole streams, indexes and bf16 decodes."""
    from weights_hq_encode_gb300 import inputs as I
    C = I.WEIGHTS8B
    cal = calibration()["weights_8b"]["E8"]
    mask = oracle.make_signs(C["sign_seed"], 0).reshape(1, 4)
    signs = torch.from_numpy(mask.view(np.int32).copy()).cuda()
    for i in range(len(C["shapes"])):
        c = cal[rate][i]
        xt = hq.as_tiles(I.weight_matrix(i, "cuda"))
        n = xt.shape[0]
        p = hq.make_params(8, c["k"], c["alpha"], 0, 0, signs, 1 << 40)
        P = oracle.make_params(8, c["k"], c["alpha"], 0, 0, mask, 1 << 40)
        stream, offsets, total = _whole(hq, oracle, xt, n, P, p)
        bps = (total * 32 - 15.5 * hq.hq_num_groups(n)) / (n * 128)
        assert abs(bps - float(rate)) < 0.01, (rate, i, bps)
        del xt, stream, offsets


@pytest.mark.parametrize("name,lat", [("Z", 1), ("A2", 2), ("D4", 4), ("E8", 8)])
def test_long_context_sweep_whole(hq, oracle, name, lat):
    """One layer's K and V of 131072 tokens, dither on, every rate of the
    sweep (1.7, 2.0, 2.5, 3.0 bps): whole streams, indexes and bf16 decodes."""
    from weights_hq_encode_gb300 import inputs as I
    C = I.LONGCTX
    cal = calibration()["long_context"]
    xt = hq.as_tiles(I.long_context_layer("cuda"))
    n = xt.shape[0]
    mask = (oracle.make_signs(C["sign_seed"], 0) ^ oracle.make_signs(C["layer_sign_seed"], 0))
    mask = mask.reshape(1, 4)
    signs = torch.from_numpy(mask.view(np.int32).copy()).cuda()
    for rate in ("1.7", "2.0", "2.5", "3.0"):
        c = cal[name][rate]
        p = hq.make_params(lat, c["k"], c["alpha"], 1, C["dither_seed"], signs, 1 << 40)
        P = oracle.make_params(lat, c["k"], c["alpha"], 1, C["dither_seed"], mask, 1 << 40)
        stream, offsets, total = _whole(hq, oracle, xt, n, P, p)
        bps = (total * 32 - 15.5 * hq.hq_num_groups(n)) / (n * 128)
        assert abs(bps - float(rate)) < 0.01, (name, rate, bps)
        del stream, offsets


@pytest.mark.parametrize("name,lat,rate", [("E8", 8, "3.0"), ("D4", 4, "2.0")])
def test_long_context_dense_rotation_whole(hq, oracle, name, lat, rate):
    """The per-layer Haar (QJL) rotation on a whole workload: the long-context
    layer with one Haar matrix for its K half and one for its V half (segments
    of 1 048 576 tiles), dither on; every stream word, index entry and bf16
    decoded value equals the oracle's fixed-order fp32 chains."""
    from weights_hq_encode_gb300 import inputs as I
    C = I.LONGCTX
    cal = calibration()["long_context"][name][rate]
    xt = hq.as_tiles(I.long_context_layer("cuda"))
    n = xt.shape[0]
    mask = (oracle.make_signs(C["sign_seed"], 0) ^ oracle.make_signs(C["layer_sign_seed"], 0))
    masks = np.stack([mask, mask])
    tps = n // 2
    rot = I.haar_rotations(2, seed=321)
    signs = torch.from_numpy(masks.view(np.int32).copy()).cuda()
    p = hq.make_params(lat, cal["k"], cal["alpha"], 1, C["dither_seed"], signs, tps,
                       rot=torch.from_numpy(rot.copy()).cuda())
    P = oracle.make_params(lat, cal["k"], cal["alpha"], 1, C["dither_seed"], masks, tps, rot=rot)
    _whole(hq, oracle, xt, n, P, p)


def test_indices_past_two_to_the_31_elements(hq, oracle):
    """A ragged input of 2^24 + 37 tiles (2^31 + 4736 elements, 4 GiB of bf16):
    the groups at the start, on both sides of element 2^31 and at the
    ragged end, and a few drawn at random, are coded and decoded exactly as
    the oracle codes each of them alone (64-bit tile, element and stream
    positions); the index is non-decreasing and ends at the stream's length."""
    n = (1 << 24) + 37
    gen = torch.Generator(device="cuda").manual_seed(31)
    xt = torch.empty(n, 128, dtype=torch.bfloat16, device="cuda")
    for a in range(0, n, 1 << 22):
        b = min(n, a + (1 << 22))
        xt[a:b] = torch.randn(b - a, 128, generator=gen, device="cuda").to(torch.bfloat16)
    cal = calibration()["kv_cache_8b"]["E8"]["3.0"]
    seed = 77
    mask = oracle.make_signs(5, 0).reshape(1, 4)
    signs = torch.from_numpy(mask.view(np.int32).copy()).cuda()
    p = hq.make_params(8, cal["k"], cal["alpha"], 1, seed, signs, n)
    stream, offsets, status, total, _ = gpu_encode(hq, p, xt, n)
    assert status == 0
    off = offsets.cpu().numpy().view(np.uint64)
    assert off[0] == 0 and off[-1] == total and (np.diff(off.astype(np.int64)) >= 0).all()
    out, st = gpu_decode(hq, p, stream, total, offsets, n, hq.HQ_OUT_BF16)
    assert st == 0
    ng = hq.hq_num_groups(n)
    edge = (1 << 24) // 32                           # the group that starts at element 2^31
    rng = np.random.default_rng(3)
    for g in sorted({0, edge - 1, edge, ng - 1} | set(rng.integers(0, ng, 4).tolist())):
        t0, t1 = 32 * g, min(n, 32 * g + 32)
        xb = xt[t0:t1].cpu().view(torch.int16).numpy().view(np.uint16)
        P = oracle.make_params(8, cal["k"], cal["alpha"], 1, seed, mask, 1 << 40, t0)
        ref = oracle.encode(P, xb)
        assert ref["status"] == 0
        words = u32(stream[int(off[g]):int(off[g + 1])])
        assert words.size == ref["total_words"] and (words == ref["stream"][:words.size]).all()
        dref = oracle.decode(P, ref["stream"], ref["offsets"], t1 - t0, out="bf16")
        got = out[t0:t1].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, dref["out"])


# ---------------------------------------------------------------- fused scores
def _scores_case(hq, oracle, n_kv, T, B, Hq, seed_tok):
    from weights_hq_encode_gb300 import inputs as I
    C = I.SCORES
    cal = calibration()["kv_cache_8b"]["E8"]["3.0"]
    K = I.scores_keys("cuda", tokens=T)[:n_kv]
    q = I.scores_queries("cuda", batch=B, q_heads=Hq)
    mask = (oracle.make_signs(C["sign_seed"], 0) ^ oracle.make_signs(C["layer_sign_seed"], 0))
    mask = mask.reshape(1, 4)
    signs = torch.from_numpy(mask.view(np.int32).copy()).cuda()
    n = n_kv * T
    p = hq.make_params(8, cal["k"], cal["alpha"], 1, seed_tok, signs, n)
    xt = hq.as_tiles(K)
    stream, offsets, status, total, _ = gpu_encode(hq, p, xt, n)
    assert status == 0
    scores = torch.full((B, Hq, T), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(hq.hq_decode_qk_workspace_bytes(B, Hq), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hq.hq_decode_qk(p, stream, total, offsets, n_kv, T, q.view(torch.int16), B, Hq, scores,
                         ws, st)
    assert rc == hq.HQ_OK
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return K, q, p, stream, offsets, total, scores, mask, cal


@pytest.mark.parametrize("n_kv,T,B,Hq", [(2, 200, 3, 8), (2, 200, 20, 8), (3, 77, 1, 3)])
def test_decode_qk_against_oracle_scores(hq, oracle, n_kv, T, B, Hq):
    """Heads that start inside a group (T not a multiple of 32), more query
    rows per head than one 64-row tile (20 x 4 = 80), one row per head."""
    K, q, p, stream, offsets, total, scores, mask, cal = _scores_case(hq, oracle, n_kv, T, B, Hq,
                                                                      500)
    P = oracle.make_params(8, cal["k"], cal["alpha"], 1, 500, mask, n_kv * T)
    ref = oracle.encode(P, K.reshape(-1, 128).cpu().view(torch.int16).numpy().view(np.uint16))
    assert (u32(stream[:total]) == ref["stream"]).all()
    khat = oracle.decode(P, ref["stream"], ref["offsets"], n_kv * T)["out"]
    qb = q.cpu().view(torch.int16).numpy().view(np.uint16)
    sref = oracle.scores(khat, n_kv, T, qb, B, Hq)
    got = scores.cpu().numpy()
    qn = np.linalg.norm((qb.astype(np.uint32) << 16).view(np.float32), axis=-1)   # [B,Hq]
    kn = np.linalg.norm(khat.reshape(n_kv, T, 128), axis=-1)                      # [n_kv,T]
    G = Hq // n_kv
    bound = 1e-4 * qn[:, :, None] * np.repeat(kn, G, axis=0)[None]
    assert np.all(np.abs(got - sref) <= bound)


def test_decode_qk_full_size_sampled(hq, oracle):
    """Fused scores on the full workload (8 heads x 32768 tokens, batch 16 x 32
    heads); a sample of tokens is checked against the oracle's decode."""
    from weights_hq_encode_gb300 import inputs as I
    C = I.SCORES
    K, q, p, stream, offsets, total, scores, mask, cal = _scores_case(
        hq, oracle, C["kv_heads"], C["tokens"], C["batch"], C["q_heads"], C["dither_seeds"][0])
    n = C["kv_heads"] * C["tokens"]
    # the whole compressed K stream and index equal the oracle's
    P = oracle.make_params(8, cal["k"], cal["alpha"], 1, C["dither_seeds"][0], mask, n)
    ref = oracle.encode(P, hq.as_tiles(K).cpu().numpy().view(np.uint16))
    assert total == ref["total_words"]
    assert (u32(stream[:total]) == ref["stream"]).all()
    assert (offsets.cpu().numpy().view(np.uint64) == ref["offsets"]).all()
    rng = np.random.default_rng(9)
    ng = hq.hq_num_groups(n)
    qb = q.cpu().view(torch.int16).numpy().view(np.uint16)
    qf = (qb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    G = C["q_heads"] // C["kv_heads"]
    for g in [0, ng - 1] + rng.integers(0, ng, 8).tolist():
        t0 = 32 * g
        xb = hq.as_tiles(K)[t0:t0 + 32].cpu().numpy().view(np.uint16)
        P = oracle.make_params(8, cal["k"], cal["alpha"], 1, C["dither_seeds"][0], mask, 1 << 40, t0)
        ref = oracle.encode(P, xb)
        khat = oracle.decode(P, ref["stream"], ref["offsets"], 32)["out"].astype(np.float64)
        for j in range(32):
            tile = t0 + j
            h, tok = tile // C["tokens"], tile % C["tokens"]
            rows = qf[:, h * G:(h + 1) * G, :]                                # [B, G, 128]
            sref = rows @ khat[j]
            got = scores[:, h * G:(h + 1) * G, tok].cpu().numpy()
            bound = 1e-4 * np.linalg.norm(rows, axis=-1) * np.linalg.norm(khat[j])
            assert np.all(np.abs(got - sref) <= bound)


def test_decode_qk_query_rows_of_very_different_magnitude(hq, oracle):
    """Query rows scaled by powers of two from 2^-100 to 2^100 (exact in
    bf16): every row's scores stay within the relative bound of its own norm,
    so the tensor-core operands keep each row's precision at any scale (a
    16-bit operand format without per-row scaling would overflow or lose the
    small rows)."""
    n_kv, T, B, Hq = 2, 200, 5, 8
    K, q, p, stream, offsets, total, scores, mask, cal = _scores_case(hq, oracle, n_kv, T, B, Hq,
                                                                      700)
    f = torch.exp2(torch.tensor([-100.0, -20.0, 0.0, 20.0, 100.0], device="cuda"))[:, None, None]
    qs = (q.float() * f).to(torch.bfloat16)
    assert torch.equal(qs.float(), q.float() * f)
    sc = torch.full((B, Hq, T), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(hq.hq_decode_qk_workspace_bytes(B, Hq), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_decode_qk(p, stream, total, offsets, n_kv, T, qs.view(torch.int16), B, Hq, sc,
                           ws, st) == hq.HQ_OK
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    P = oracle.make_params(8, cal["k"], cal["alpha"], 1, 700, mask, n_kv * T)
    ref = oracle.encode(P, K.reshape(-1, 128).cpu().view(torch.int16).numpy().view(np.uint16))
    khat = oracle.decode(P, ref["stream"], ref["offsets"], n_kv * T)["out"]
    qb = qs.cpu().view(torch.int16).numpy().view(np.uint16)
    sref = oracle.scores(khat, n_kv, T, qb, B, Hq)
    qn = np.linalg.norm((qb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=-1)
    kn = np.linalg.norm(khat.reshape(n_kv, T, 128).astype(np.float64), axis=-1)
    bound = 1e-4 * qn[:, :, None] * np.repeat(kn, Hq // n_kv, axis=0)[None]
    assert np.all(np.abs(sc.cpu().numpy().astype(np.float64) - sref) <= bound)


def test_decode_qk_corrupt_group_scores_zero(hq, oracle):
    """A corrupt group of the compressed K (its index entry points past the
    next group) is flagged and its tokens score 0 for every query row, as if
    its keys decoded to zeros; every other token's score is unchanged."""
    n_kv, T, B, Hq = 2, 200, 3, 8
    K, q, p, stream, offsets, total, scores, mask, cal = _scores_case(hq, oracle, n_kv, T, B, Hq,
                                                                      600)
    good = scores.clone()
    bad_off = offsets.clone()
    bad_off[4] = bad_off[5] + 1                       # group 3 now ends past group 4's start
    sc = torch.full_like(scores, 7.0)
    ws = torch.empty(hq.hq_decode_qk_workspace_bytes(B, Hq), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_decode_qk(p, stream, total, bad_off, n_kv, T, q.view(torch.int16), B, Hq, sc,
                           ws, st) == hq.HQ_OK
    torch.cuda.synchronize()
    assert int(st.item()) & hq.HQ_ERR_CORRUPT
    tiles = np.arange(n_kv * T)
    g = tiles // 32
    hit = (g == 3) | (g == 4)                          # the groups whose bounds changed
    G = Hq // n_kv
    got, ref = sc.cpu().numpy(), good.cpu().numpy()
    for h in range(n_kv):
        tok = np.arange(T)
        hh = hit[h * T + tok]
        rows = slice(h * G, (h + 1) * G)
        assert (got[:, rows][:, :, hh] == 0).all()
        assert (got[:, rows][:, :, ~hh] == ref[:, rows][:, :, ~hh]).all()

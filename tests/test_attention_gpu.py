"""GPU parity of decode attention over compressed K and V (closing section of
the HyperQuant summary: fused decode + MMA) against the fp64 oracle
(oracle/attention.py) on the oracle's own decodes.

The K and V streams are written by the CPU oracle and copied to the GPU, so
every expected value comes from the oracle alone.

Tolerance, derived to first order in u = 2^-24 from the fp32 steps of the
CUDA path.  A score is the rotated query (7 rounded transform stages and one
scaling: 8 u) dotted with e on the tensor cores: the query row and the
token are each scaled by a power of two to below 1 (exact) and split into
two fp16 parts (per value |x - x_1 - x_2| <= 2^-22 |x| + 2^-25, the second
term from fp16's subnormal spacing), and the three kept partial products
q_1 e_1 + q_1 e_2 + q_2 e_1 miss the exact dot of the scaled vectors x, y
by at most 3 * 2^-22 sum|x_i y_i| + 2^-25 (sum|x_i| + sum|y_i|) <= 35 u |x| |y|
(the largest scaled value is at least 1/2 and sum|x_i| <= sqrt(128) |x|),
i.e. 35 u |q'| |e_t| once the scales are undone; they
are accumulated in fp32 over 24 MMA steps, at most 2 u each even if the
accumulation truncates (48 u).  So |dz_t| <= (8 + 35 + 48) u zeta <
136 u zeta, zeta = scale |q| max_t |Khat_t| (the transform is orthogonal,
so |q'| |e_t| = |q| |Khat_t|).  Softmax turns that into a relative error of
p_t of at most 2 max|dz| plus a few u for exp and the division.  The value
side sums p_t e_t over at most 256 tokens per chunk on the tensor cores:
both operands split into two tf32 parts (|x - hi - lo| <= 2^-22 |x| = 4 u |x|,
so each product of the parts is within 8 u of p_t e_t), the products exact,
accumulated in fp32 tensor memory over 64 MMA steps per chunk (2 u per step
even if the accumulation truncates: 128 u), the two halves of the split
added once (u), then 129 chunks per head combined in fp32 (129 u): together
(8 + 128 + 1 + 129) u < 400 u relative to sum_t p_t |Vhat_t,d|.  So an
element of out is held to (2 * 136 u zeta + 600 u) of sum_t p_t |Vhat_t,d|,
i.e. (1.7e-5 zeta + 3.6e-5), and p_t to (1.7e-5 zeta + 1e-6) of p_t plus
1e-38 for values below the fp32 normal range."""
import numpy as np
import pytest
import torch

from _cases import calibration

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq as H
    return H


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.reshape(-1, 128).cpu().view(torch.int16).numpy().view(np.uint16)


class Side:
    """One compressed stream (K or V), written and decoded by the oracle."""

    def __init__(self, oracle, hq, x_bits, lattice, k, alpha, seed, mask, tps, rot=None):
        self.P = oracle.make_params(lattice, k, alpha, 1, seed, mask, tps, rot=rot)
        enc = oracle.encode(self.P, x_bits)
        assert enc["status"] == 0
        self.words = int(enc["total_words"])
        self.hat = oracle.decode(self.P, enc["stream"], enc["offsets"], x_bits.shape[0])["out"]
        s = np.ascontiguousarray(enc["stream"][:max(self.words, 1)]).view(np.int32)
        self.stream = torch.from_numpy(s.copy()).cuda()
        self.offsets = torch.from_numpy(np.ascontiguousarray(enc["offsets"]).view(np.int64).copy()).cuda()
        signs = torch.from_numpy(np.ascontiguousarray(mask, dtype=np.uint32).view(np.int32).copy()).cuda()
        self.rot = None if rot is None else torch.from_numpy(np.ascontiguousarray(rot)).cuda()
        self.p = hq.make_params(lattice, k, alpha, 1, seed, signs, tps, rot=self.rot)


def _masks(oracle, layer_seed):
    from weights_hq_encode_gb300 import inputs as I
    C = I.SCORES
    return (oracle.make_signs(C["sign_seed"], 0) ^ oracle.make_signs(layer_seed, 0)).reshape(1, 4)


def _run(hq, Ks, Vs, n_kv, T, q_bits, B, Hq, scale, probs=True):
    q = torch.from_numpy(q_bits.view(np.int16).copy()).cuda()
    out = torch.full((B, Hq, 128), 7.0, dtype=torch.float32, device="cuda")
    pr = torch.full((B, Hq, T), 7.0, dtype=torch.float32, device="cuda") if probs else None
    ws = torch.empty(hq.hq_decode_attention_workspace_bytes(n_kv, T, B, Hq), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hq.hq_decode_attention(Ks.p, Ks.stream, Ks.words, Ks.offsets, Vs.p, Vs.stream, Vs.words,
                                Vs.offsets, n_kv, T, q, B, Hq, scale, out, pr, ws, st)
    assert rc == hq.HQ_OK
    torch.cuda.synchronize()
    return out.cpu().numpy(), (pr.cpu().numpy() if probs else None), int(st.item())


def _check(A, Ks, Vs, n_kv, T, q_bits, B, Hq, scale, out, probs, rot=False):
    ref, P = A.attention(Ks.hat, Vs.hat, q_bits, n_kv, T, B, Hq, scale)
    G = Hq // n_kv
    V = np.abs(Vs.hat.astype(np.float64)).reshape(n_kv, T, 128)
    size = np.stack([np.einsum("bgt,td->bgd", P[:, h * G:(h + 1) * G], V[h]) for h in range(n_kv)],
                    axis=1).reshape(B, Hq, 128)
    qn = np.linalg.norm(A.bf16_bits_to_f64(q_bits), axis=-1)                      # [B, Hq]
    kmax = np.linalg.norm(Ks.hat.astype(np.float64).reshape(n_kv, T, 128), axis=-1).max(-1)
    zeta = scale * qn * np.repeat(kmax, G)[None, :]                                # [B, Hq]
    # a dense rotation adds one more 128-term chain on each side: R_K q doubles
    # the score term, and R_V^T on the output row adds 128 u |out row|
    tol = ((3.4e-5 if rot else 1.7e-5) * zeta + 3.6e-5)[:, :, None]
    if rot:
        tol = tol + 128 * 2.0 ** -24 * np.linalg.norm(ref, axis=-1, keepdims=True) / (size + 1e-30)
    err = np.abs(out - ref) / (size + 1e-30)
    worst = np.unravel_index(np.argmax(err / tol), err.shape)
    assert np.all(err <= tol), (err[worst], zeta[worst[:2]], tol[worst[0], worst[1], 0])
    if probs is not None:
        tolp = ((3.4e-5 if rot else 1.7e-5) * zeta + 1e-6)[:, :, None]
        assert np.all(np.abs(probs - P) <= tolp * P + 1e-38)
    return (err / tol).max()


def _workload(oracle, hq, n_kv, T, B, Hq, lat_k=8, lat_v=8, rot=False):
    from weights_hq_encode_gb300 import inputs as I
    C = I.SCORES
    cal = calibration()
    other = {4: cal["long_context"]["D4"]["2.5"], 1: cal["long_context"]["Z"]["2.0"],
             2: dict(k=1, alpha=cal["long_context"]["D4"]["2.5"]["alpha"])}
    ck = cal["kv_cache_8b"]["E8"]["3.0"] if lat_k == 8 else other[lat_k]
    cv = cal["kv_cache_8b"]["E8"]["2.0"] if lat_v == 8 else other[lat_v]
    kb = _bits(I.scores_keys("cpu", tokens=T)[:n_kv])
    vb = _bits(I.scores_values("cpu", tokens=T)[:n_kv])
    n = n_kv * T
    Rk = I.haar_rotations(1, seed=31) if rot else None
    Rv = I.haar_rotations(1, seed=32) if rot else None
    Ks = Side(oracle, hq, kb, lat_k, ck["k"], ck["alpha"], C["dither_seeds"][0],
              _masks(oracle, C["layer_sign_seed"]), n, rot=Rk)
    Vs = Side(oracle, hq, vb, lat_v, cv["k"], cv["alpha"], C["dither_seeds"][1],
              _masks(oracle, C["layer_sign_seed"] + 1), n, rot=Rv)
    q_bits = _bits(I.scores_queries("cpu", batch=B, q_heads=Hq)).reshape(B, Hq, 128)
    return Ks, Vs, q_bits


@pytest.mark.parametrize("n_kv,T,B,Hq,lat_k,lat_v", [
    (2, 100, 3, 6, 8, 8),        # groups straddle the two heads (T not a multiple of 32)
    (2, 64, 20, 8, 8, 8),        # 80 query rows per head: two row tiles
    (1, 1, 1, 1, 8, 8),          # one token
    (3, 700, 2, 6, 4, 1),        # D4 keys, Z values
    (2, 160, 2, 4, 2, 2),        # A2 keys and values
])
def test_attention_against_oracle(hq, oracle, n_kv, T, B, Hq, lat_k, lat_v):
    from oracle import attention as A
    Ks, Vs, q_bits = _workload(oracle, hq, n_kv, T, B, Hq, lat_k, lat_v)
    scale = 128 ** -0.5
    out, probs, st = _run(hq, Ks, Vs, n_kv, T, q_bits, B, Hq, scale)
    assert st == 0
    _check(A, Ks, Vs, n_kv, T, q_bits, B, Hq, scale, out, probs)
    out2, _, st2 = _run(hq, Ks, Vs, n_kv, T, q_bits, B, Hq, scale, probs=False)
    assert st2 == 0 and np.array_equal(out, out2)             # deterministic


@pytest.mark.parametrize("n_kv,T,B,Hq", [(2, 96, 3, 6), (1, 320, 2, 4)])
def test_attention_with_dense_rotation(hq, oracle, n_kv, T, B, Hq):
    """K and V coded with per-layer Haar (QJL) rotations: the queries are
    rotated by R_K and the output rows by R_V^T."""
    from oracle import attention as A
    Ks, Vs, q_bits = _workload(oracle, hq, n_kv, T, B, Hq, rot=True)
    out, probs, st = _run(hq, Ks, Vs, n_kv, T, q_bits, B, Hq, 128 ** -0.5)
    assert st == 0
    _check(A, Ks, Vs, n_kv, T, q_bits, B, Hq, 128 ** -0.5, out, probs, rot=True)


def test_attention_full_size(hq, oracle):
    """The decode-attention workload: 8 KV heads x 32768 tokens, batch 16 x 32
    query heads, K at 3 bps and V at 2 bps (E8)."""
    from oracle import attention as A
    from weights_hq_encode_gb300 import inputs as I
    C = I.SCORES
    n_kv, T, B, Hq = C["kv_heads"], C["tokens"], C["batch"], C["q_heads"]
    Ks, Vs, q_bits = _workload(oracle, hq, n_kv, T, B, Hq)
    out, probs, st = _run(hq, Ks, Vs, n_kv, T, q_bits, B, Hq, 128 ** -0.5)
    assert st == 0
    _check(A, Ks, Vs, n_kv, T, q_bits, B, Hq, 128 ** -0.5, out, probs)


def test_attention_corrupt_value_stream_is_flagged(hq, oracle):
    n_kv, T, B, Hq = 2, 96, 2, 4
    Ks, Vs, q_bits = _workload(oracle, hq, n_kv, T, B, Hq)
    Vs.offsets[1] = Vs.offsets[2] + 1                        # group 0 now ends past group 1
    out, _, st = _run(hq, Ks, Vs, n_kv, T, q_bits, B, Hq, 0.1, probs=False)
    assert st & hq.HQ_ERR_CORRUPT
    assert np.isfinite(out).all()


def test_attention_invalid_arguments(hq, oracle):
    n_kv, T, B, Hq = 2, 64, 2, 4
    Ks, Vs, q_bits = _workload(oracle, hq, n_kv, T, B, Hq)
    q = torch.from_numpy(q_bits.view(np.int16).copy()).cuda()
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(hq.hq_decode_attention_workspace_bytes(n_kv, T, B, Hq), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_decode_attention_workspace_bytes(3, T, B, Hq) == 0     # Hq % n_kv != 0
    args = [Ks.p, Ks.stream, Ks.words, Ks.offsets, Vs.p, Vs.stream, Vs.words, Vs.offsets]
    assert hq.hq_decode_attention(*args, 3, T, q, B, Hq, 0.1, out, None, ws, st) == hq.HQ_ERR_INVALID
    assert hq.hq_decode_attention(*args, n_kv, T, q, B, Hq, 0.1, out, None, ws[:16], st) == hq.HQ_ERR_INVALID
    assert hq.hq_decode_attention(*args, n_kv, T, None, B, Hq, 0.1, out, None, ws, st) == hq.HQ_ERR_INVALID

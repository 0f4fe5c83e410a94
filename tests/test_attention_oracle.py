"""Pins of the decode-attention oracle (no GPU).

Each check ties oracle/attention.py to a value fixed by the mathematics, not
to a second copy of its own formula: a single token, a zero query and equal
keys have closed forms; two tokens follow the logistic function; the output
is a convex combination; per-head constant values expose the query-head to
KV-head mapping; token order does not matter."""
import math

import numpy as np

from oracle import attention as A


def _bits(x):
    """fp64 values that are exact in bf16 -> bf16 bit patterns."""
    f = np.asarray(x, dtype=np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(A.bf16_bits_to_f64(b), np.asarray(x, dtype=np.float64))
    return b


def _rand(rng, *shape, scale=1.0):
    # bf16-exact values: small integers times a power of two
    return rng.integers(-64, 65, size=shape).astype(np.float64) * scale / 16.0


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    K, V = _rand(rng, 2, 128), _rand(rng, 2, 128)
    q = _bits(_rand(rng, 3, 4, 128))
    out, P = A.attention(K, V, q, 2, 1, 3, 4, 0.3)
    assert np.all(P == 1.0)
    for hq in range(4):
        assert np.array_equal(out[:, hq], np.broadcast_to(V[hq // 2], (3, 128)))


def test_zero_query_and_equal_keys_average_the_values():
    rng = np.random.default_rng(2)
    T = 37
    V = _rand(rng, T, 128)
    K = _rand(rng, T, 128)
    out, P = A.attention(K, V, _bits(np.zeros((1, 1, 128))), 1, T, 1, 1, 0.7)
    assert np.allclose(P, 1.0 / T, rtol=1e-15, atol=0)
    assert np.allclose(out[0, 0], V.mean(0), rtol=1e-13, atol=1e-15)
    Keq = np.broadcast_to(K[0], (T, 128))
    out2, _ = A.attention(Keq, V, _bits(_rand(rng, 1, 1, 128)), 1, T, 1, 1, 0.7)
    assert np.allclose(out2[0, 0], V.mean(0), rtol=1e-13, atol=1e-15)


def test_two_tokens_follow_the_logistic_function():
    rng = np.random.default_rng(3)
    K, V = _rand(rng, 2, 128), _rand(rng, 2, 128)
    q = _rand(rng, 1, 1, 128)
    scale = 0.125
    out, P = A.attention(K, V, _bits(q), 1, 2, 1, 1, scale)
    d = scale * (sum(K[1, i] * q[0, 0, i] for i in range(128)) -
                 sum(K[0, i] * q[0, 0, i] for i in range(128)))
    p0 = 1.0 / (1.0 + math.exp(d))
    assert abs(P[0, 0, 0] - p0) <= 1e-15 and abs(P[0, 0, 1] - (1 - p0)) <= 1e-15
    assert np.allclose(out[0, 0], p0 * V[0] + (1 - p0) * V[1], rtol=1e-13, atol=1e-14)


def test_output_is_a_convex_combination_and_order_free():
    rng = np.random.default_rng(4)
    n_kv, T, B, Hq = 2, 50, 2, 6
    K = rng.standard_normal((n_kv * T, 128)) * 3
    V = rng.standard_normal((n_kv * T, 128))
    q = _bits(_rand(rng, B, Hq, 128))
    out, P = A.attention(K, V, q, n_kv, T, B, Hq, 128 ** -0.5)
    assert np.allclose(P.sum(-1), 1.0, rtol=0, atol=1e-14) and (P >= 0).all()
    for hq in range(Hq):
        h = hq // (Hq // n_kv)
        Vh = V[h * T:(h + 1) * T]
        assert (out[:, hq] <= Vh.max(0) + 1e-12).all() and (out[:, hq] >= Vh.min(0) - 1e-12).all()
    perm = np.concatenate([h * T + rng.permutation(T) for h in range(n_kv)])
    out_p, _ = A.attention(K[perm], V[perm], q, n_kv, T, B, Hq, 128 ** -0.5)
    assert np.allclose(out_p, out, rtol=1e-12, atol=1e-14)


def test_query_heads_read_their_own_kv_head():
    rng = np.random.default_rng(5)
    n_kv, T, B, Hq = 4, 9, 2, 8                     # G = 2: heads 2h, 2h+1 read head h
    K = rng.standard_normal((n_kv * T, 128))
    V = np.repeat(np.arange(1, n_kv + 1, dtype=np.float64), T)[:, None] * np.ones((1, 128))
    out, _ = A.attention(K, V, _bits(_rand(rng, B, Hq, 128)), n_kv, T, B, Hq, 0.2)
    for hq in range(Hq):
        assert np.allclose(out[:, hq], hq // 2 + 1, rtol=0, atol=1e-13)

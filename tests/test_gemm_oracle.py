"""Pins of the compressed-weight product oracle (no GPU).

oracle/gemm.py is tied to facts of the mathematics rather than to a second
copy of its own formula: a unit activation selects one column of the decoded
matrix, the product is linear in x, the row-major tile order puts tile t at
row t // (cols / 128), and a permutation of the input features applied to
both operands changes nothing."""
import numpy as np
import pytest

from oracle import gemm as M


def _bits(x):
    f = np.asarray(x, dtype=np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(M.bf16_bits_to_f64(b), np.asarray(x, dtype=np.float64))
    return b


def _rand_exact(rng, *shape):
    return rng.integers(-64, 65, size=shape).astype(np.float64) / 16.0


def test_unit_activation_selects_a_column():
    rng = np.random.default_rng(1)
    rows, cols = 5, 256
    W = rng.standard_normal((rows, cols))
    tiles = W.reshape(-1, 128)
    for i in (0, 127, 128, 255):
        x = np.zeros((1, cols))
        x[0, i] = 1.0
        y = M.gemm(tiles, _bits(x), rows, cols)
        assert np.array_equal(y[0], W[:, i])


def test_tile_order_is_row_major():
    rows, cols = 3, 384                                   # 3 tiles per row
    tiles = np.repeat(np.arange(rows * cols // 128, dtype=np.float64), 128).reshape(-1, 128)
    y = M.gemm(tiles, _bits(np.ones((1, cols))), rows, cols)
    # row o holds tiles 3o, 3o+1, 3o+2, each 128 copies of its index
    assert np.array_equal(y[0], [128 * (3 * o + 3 * o + 1 + 3 * o + 2) for o in range(rows)])


def test_linear_in_the_activations():
    rng = np.random.default_rng(2)
    rows, cols = 7, 512
    tiles = rng.standard_normal((rows * cols // 128, 128))
    x1, x2 = _rand_exact(rng, 2, cols), _rand_exact(rng, 2, cols)
    y1, y2 = M.gemm(tiles, _bits(x1), rows, cols), M.gemm(tiles, _bits(x2), rows, cols)
    y12 = M.gemm(tiles, _bits(x1 + 0.5 * x2), rows, cols)
    assert np.allclose(y12, y1 + 0.5 * y2, rtol=1e-12, atol=1e-12)


def test_feature_permutation_invariance():
    rng = np.random.default_rng(3)
    rows, cols = 4, 256
    W = rng.standard_normal((rows, cols))
    x = _rand_exact(rng, 3, cols)
    perm = rng.permutation(cols)
    y = M.gemm(W.reshape(-1, 128), _bits(x), rows, cols)
    yp = M.gemm(W[:, perm].reshape(-1, 128), _bits(x[:, perm]), rows, cols)
    assert np.allclose(y, yp, rtol=1e-12, atol=1e-12)


def test_rejects_ragged_columns():
    with pytest.raises(ValueError):
        M.gemm(np.zeros((1, 128)), np.zeros((1, 100), np.uint16), 1, 100)

"""Pins of the per-layer dense (Haar / QJL) rotation in the oracle (no GPU).

HyperQuant summary, Method 3-4: the per-layer rotation is a full
Haar-uniform QJL matrix or the cheap +-1 diagonal.  The oracle's dense path
(tile coded as RHT(R x), decoded as R^T applied after the inverse) is tied to
exact special cases: the identity changes nothing; a permutation codes the
permuted tile (which also fixes R before the sign diagonal); a +-1 diagonal
equals the same signs folded into the mask; and a Haar matrix keeps the
round-trip error of the unrotated codec."""
import numpy as np
import pytest


def _tiles(n=96, seed=3):
    from weights_hq_encode_gb300 import inputs as I
    x = I.bf16_bits(I.tiny_kv())
    return np.concatenate([x] * (n // x.shape[0] + 1))[:n].reshape(-1, 128)


def _enc_dec(oracle, x, mask, rot=None, lattice=8, k=2, alpha=1.7, tps=1 << 40):
    P = oracle.make_params(lattice, k, alpha, 1, 5, mask, tps, rot=rot)
    enc = oracle.encode(P, x, want_codes=True)
    dec = oracle.decode(P, enc["stream"], enc["offsets"], x.shape[0])
    return enc, dec


def test_identity_rotation_changes_nothing(oracle):
    x = _tiles()
    m = oracle.make_signs(9, 0).reshape(1, 4)
    e0, d0 = _enc_dec(oracle, x, m)
    e1, d1 = _enc_dec(oracle, x, m, rot=np.eye(128, dtype=np.float32)[None])
    assert np.array_equal(e0["stream"], e1["stream"]) and np.array_equal(d0["out"], d1["out"])


def test_permutation_codes_the_permuted_tile(oracle):
    rng = np.random.default_rng(4)
    x = _tiles()
    n_seg = 3
    tps = 32
    masks = np.stack([oracle.make_signs(9, s) for s in range(n_seg)])
    perms = [rng.permutation(128) for _ in range(n_seg)]
    R = np.stack([np.eye(128, dtype=np.float32)[p] for p in perms])      # (R x)_i = x[p[i]]
    xp = np.stack([x[t][perms[t // tps]] for t in range(x.shape[0])])
    e1, d1 = _enc_dec(oracle, x, masks, rot=R, tps=tps)
    e0, d0 = _enc_dec(oracle, xp, masks, tps=tps)
    assert np.array_equal(e1["codes"], e0["codes"])
    for t in range(x.shape[0]):                                          # x_hat = R^T (decode of R x)
        inv = np.empty(128, np.int64)
        inv[perms[t // tps]] = np.arange(128)
        assert np.array_equal(d1["out"][t], d0["out"][t][inv])


def test_sign_diagonal_equals_the_folded_mask(oracle):
    x = _tiles()
    m = oracle.make_signs(9, 0)
    s = oracle.make_signs(10, 0)
    bits = ((s[np.arange(128) >> 5] >> (np.arange(128) & 31)) & 1).astype(np.float32)
    R = np.diag(1.0 - 2.0 * bits).astype(np.float32)[None]
    e1, d1 = _enc_dec(oracle, x, m.reshape(1, 4), rot=R)
    e0, d0 = _enc_dec(oracle, x, (m ^ s).reshape(1, 4))
    assert np.array_equal(e1["stream"], e0["stream"]) and np.array_equal(d1["out"], d0["out"])


def test_haar_rotation_keeps_the_round_trip_error(oracle):
    from weights_hq_encode_gb300 import inputs as I
    R = I.haar_rotations(2)
    assert np.allclose(R[0] @ R[0].T, np.eye(128), atol=2e-6)
    x = _tiles(256)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    m = oracle.make_signs(9, 0).reshape(1, 4)
    errs = []
    for rot in (None, R[:1]):
        _, d = _enc_dec(oracle, x, m, rot=rot)
        errs.append(((d["out"] - xf) ** 2).sum() / (xf ** 2).sum())
    assert abs(errs[1] / errs[0] - 1) < 0.15, errs
    # the fixed-order chains invert each other up to fp32 rounding
    v = xf[0].astype(np.float32)
    back = oracle.rotate(R[0], oracle.rotate(R[0], v), transpose=True)
    assert np.max(np.abs(back - v)) <= 1e-5 * np.abs(v).max()

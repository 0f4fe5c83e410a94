"""GPU parity of products with a compressed weight matrix (hq_decode_gemm)
against the fp64 oracle (oracle/gemm.py) on the oracle's own decode.

The weight streams are written by the CPU oracle and copied to the GPU.
Tolerance, derived to first order in u = 2^-24 from the fp32 steps: each
tile's share is a 128-term fp32 dot of the rotated activation tile (7 rounded
transform stages and one scaling) with e, |d share_j| <= 136 u |x_j| |What_oj|
(the transform is orthogonal); the shares of a row are summed in fp32 with at
most tpr/32 sequential additions per lane plus 5 butterfly levels.  So
|dy[b][o]| <= (142 + tpr/32) u S[b][o],  S = sum_j |x_bj| |What_oj|."""
import numpy as np
import pytest
import torch

from _cases import calibration

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq as H
    return H


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _weights(oracle, hq, wb, rows, cols, lattice, k, alpha, dither, seed, rot=None):
    from weights_hq_encode_gb300 import inputs as I
    mask = oracle.make_signs(I.WEIGHTS8B["sign_seed"], 0).reshape(1, 4)
    n = rows * cols // 128
    P = oracle.make_params(lattice, k, alpha, dither, seed, mask, 1 << 40, rot=rot)
    enc = oracle.encode(P, wb.reshape(-1, 128))
    assert enc["status"] == 0
    words = int(enc["total_words"])
    what = oracle.decode(P, enc["stream"], enc["offsets"], n)["out"]
    stream = torch.from_numpy(np.ascontiguousarray(enc["stream"][:max(words, 1)]).view(np.int32).copy()).cuda()
    offsets = torch.from_numpy(np.ascontiguousarray(enc["offsets"]).view(np.int64).copy()).cuda()
    signs = torch.from_numpy(mask.astype(np.uint32).view(np.int32).copy()).cuda()
    rt = None if rot is None else torch.from_numpy(np.ascontiguousarray(rot)).cuda()
    p = hq.make_params(lattice, k, alpha, dither, seed, signs, 1 << 40, rot=rt)
    return p, stream, words, offsets, what, (signs, rt)


def _run(hq, p, stream, words, offsets, rows, cols, xb):
    B = xb.shape[0]
    x = torch.from_numpy(xb.view(np.int16).copy()).cuda()
    y = torch.full((B, rows), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(hq.hq_decode_gemm_workspace_bytes(rows, cols, B), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_decode_gemm(p, stream, words, offsets, rows, cols, x, B, y, ws, st) == hq.HQ_OK
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(st.item())


def _check(G, what, xb, rows, cols, y, rot=False):
    ref = G.gemm(what, xb, rows, cols)
    tpr = cols // 128
    xn = np.linalg.norm(G.bf16_bits_to_f64(xb).reshape(-1, tpr, 128), axis=-1)        # [B, tpr]
    wn = np.linalg.norm(what.astype(np.float64).reshape(rows, tpr, 128), axis=-1)     # [rows, tpr]
    S = xn @ wn.T
    tol = (142 + (128 if rot else 0) + tpr / 32) * U * S   # R x_j: one more 128-term chain
    assert np.all(np.abs(y - ref) <= tol), np.max(np.abs(y - ref) / (tol + 1e-300))


@pytest.mark.parametrize("index,rows,B,rate,lattice,dither", [
    (0, 64, 1, "4.0", 8, 0),      # 4096 columns: one row per group
    (2, 33, 5, "3.0", 8, 0),      # 14336 columns: rows straddle groups
    (2, 33, 16, "3.0", 8, 1),     # the same with four groups a block (ragged last blocks)
    (3, 100, 17, "5.0", 8, 1),    # 4096 columns, three batch chunks, dither on
    (1, 50, 3, "4.0", 4, 0),      # D4
    (0, 20, 2, "4.0", 1, 0),      # Z
    (1, 24, 4, "4.0", 2, 1),      # A2, dither on
])
def test_gemm_against_oracle(hq, oracle, index, rows, B, rate, lattice, dither):
    from oracle import gemm as G
    from weights_hq_encode_gb300 import inputs as I
    cols = I.WEIGHTS8B["shapes"][index][1]
    c = calibration()["weights_8b"]["E8"][rate][index]
    alpha = c["alpha"] if lattice == 8 else c["alpha"] * {4: 0.5, 2: 0.45, 1: 0.35}[lattice]
    wb = _bits(I.weight_matrix(index, "cpu", rows=rows))
    p, stream, words, offsets, what, _s = _weights(oracle, hq, wb, rows, cols, lattice, c["k"],
                                                   alpha, dither, 901)
    xb = _bits(I.activations(B, cols, device="cpu"))
    y, st = _run(hq, p, stream, words, offsets, rows, cols, xb)
    assert st == 0
    _check(G, what, xb, rows, cols, y)
    y2, _ = _run(hq, p, stream, words, offsets, rows, cols, xb)
    assert np.array_equal(y, y2)                                 # deterministic


@pytest.mark.parametrize("cols,rows,B", [(128, 37, 1), (512, 19, 9), (2048, 21, 16)])
def test_gemm_narrow_matrices(hq, oracle, cols, rows, B):
    """Matrices of 1, 4 and 16 tiles a row (the first columns of a
    Llama-shaped weight): a group of 32 tiles holds whole rows, so the
    product kernel sums each row's tile shares itself.  The row counts leave
    the last group partial; the batch sizes take one, two and four groups a
    block and a ragged chunk of activation rows."""
    from oracle import gemm as G
    from weights_hq_encode_gb300 import inputs as I
    c = calibration()["weights_8b"]["E8"]["4.0"][0]
    wb = np.ascontiguousarray(_bits(I.weight_matrix(0, "cpu", rows=rows))[:, :cols])
    p, stream, words, offsets, what, _s = _weights(oracle, hq, wb, rows, cols, 8, c["k"],
                                                   c["alpha"], 1, 5)
    xb = _bits(I.activations(B, cols, device="cpu"))
    y, st = _run(hq, p, stream, words, offsets, rows, cols, xb)
    assert st == 0
    _check(G, what, xb, rows, cols, y)


def test_gemm_with_dense_rotation(hq, oracle):
    """Weights coded with a Haar (QJL) rotation: each activation tile is
    rotated by R before the transform."""
    from oracle import gemm as G
    from weights_hq_encode_gb300 import inputs as I
    rows, cols, B = 40, 4096, 3
    c = calibration()["weights_8b"]["E8"]["4.0"][0]
    wb = _bits(I.weight_matrix(0, "cpu", rows=rows))
    p, stream, words, offsets, what, _s = _weights(oracle, hq, wb, rows, cols, 8, c["k"],
                                                   c["alpha"], 0, 0, rot=I.haar_rotations(1, 7))
    xb = _bits(I.activations(B, cols, device="cpu"))
    y, st = _run(hq, p, stream, words, offsets, rows, cols, xb)
    assert st == 0
    _check(G, what, xb, rows, cols, y, rot=True)


@pytest.mark.parametrize("index,B", [(0, 16), (2, 8)])
def test_gemm_full_matrix(hq, oracle, index, B):
    """Whole Llama-3.1-8B-shaped matrices (4096 x 4096 and 4096 x 14336) at
    4 bps with the frozen calibration."""
    from oracle import gemm as G
    from weights_hq_encode_gb300 import inputs as I
    rows, cols = I.WEIGHTS8B["shapes"][index]
    c = calibration()["weights_8b"]["E8"]["4.0"][index]
    wb = _bits(I.weight_matrix(index, "cpu"))
    p, stream, words, offsets, what, _s = _weights(oracle, hq, wb, rows, cols, 8, c["k"],
                                                   c["alpha"], 0, 0)
    xb = _bits(I.activations(B, cols, device="cpu"))
    y, st = _run(hq, p, stream, words, offsets, rows, cols, xb)
    assert st == 0
    _check(G, what, xb, rows, cols, y)


def test_gemm_invalid_arguments(hq, oracle):
    from weights_hq_encode_gb300 import inputs as I
    rows, cols, B = 8, 4096, 2
    c = calibration()["weights_8b"]["E8"]["4.0"][0]
    wb = _bits(I.weight_matrix(0, "cpu", rows=rows))
    p, stream, words, offsets, what, _s = _weights(oracle, hq, wb, rows, cols, 8, c["k"],
                                                   c["alpha"], 0, 0)
    x = torch.zeros((B, cols), dtype=torch.int16, device="cuda")
    y = torch.empty((B, rows), dtype=torch.float32, device="cuda")
    ws = torch.empty(hq.hq_decode_gemm_workspace_bytes(rows, cols, B), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_decode_gemm_workspace_bytes(rows, 100, B) == 0
    assert hq.hq_decode_gemm(p, stream, words, offsets, rows, 100, x, B, y, ws, st) == hq.HQ_ERR_INVALID
    assert hq.hq_decode_gemm(p, stream, words, offsets, rows, cols, x, B, y, ws[:64], st) == hq.HQ_ERR_INVALID
    p.tiles_per_segment = 4                                       # matrix spans several segments
    assert hq.hq_decode_gemm(p, stream, words, offsets, rows, cols, x, B, y, ws, st) == hq.HQ_ERR_INVALID

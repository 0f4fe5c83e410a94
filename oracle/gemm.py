"""Products with a compressed weight matrix: a plain fp64 reference.

Test infrastructure only (imported by tests/, __graft_entry__.smoke() and
bench.py's CPU legs); it shares nothing with the CUDA path.

HyperQuant summary, Method 2 and the closing section (weights coded with the
same tile codec; decode fused with the matrix product).  Reading: a weight
matrix W [rows, cols] (cols a multiple of 128) is coded row-major as
rows * cols / 128 tiles, tile t holding W[t // (cols/128)][128 (t % (cols/128)) :][:128];
the fused product of a batch of activations x [B, cols] (bf16) is

    y[b, o] = sum_i What[o, i] * x[b, i]

with What the decode of the stream (fp32, widened to fp64) and x widened
exactly.  numpy's matrix product serves as the inner products, in fp64.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm(what: np.ndarray, x_bits: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """y [B, rows] = x What^T in fp64.  what: [rows * cols / 128, 128] decoded
    tiles (any float dtype); x_bits: [B, cols] bf16 bit patterns."""
    if cols % 128 != 0:
        raise ValueError("cols must be a multiple of 128")
    W = np.asarray(what, dtype=np.float64).reshape(rows, cols)
    x = bf16_bits_to_f64(x_bits).reshape(-1, cols)
    return x @ W.T

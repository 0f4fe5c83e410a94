"""Decode attention over a compressed KV cache: a plain fp64 reference.

Test infrastructure only (imported by tests/, __graft_entry__.smoke() and
bench.py's CPU legs); it shares nothing with the CUDA path.

HyperQuant summary, closing section (fused decode + MMA): attention computed
straight from the compressed K and V.  Reading (the summary gives no formula):
standard scaled dot-product attention of one decode step with grouped query
heads,

    s[b, hq, t] = scale * <q[b, hq], Khat[h, t]>,   h = hq // (Hq // n_kv)
    p[b, hq, :] = softmax over t of s[b, hq, :]     (maximum subtracted first)
    out[b, hq]  = sum_t p[b, hq, t] * Vhat[h, t]

where Khat and Vhat are the decodes of the two streams (fp32, here widened
to fp64), head h's token t is tile h * n_tokens + t of its stream, and q holds
bf16 bit patterns widened exactly.  All arithmetic is fp64; numpy's dot serves
as the inner product.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention(khat: np.ndarray, vhat: np.ndarray, q_bits: np.ndarray, n_kv: int,
              n_tokens: int, B: int, Hq: int, scale: float):
    """(out [B, Hq, 128], p [B, Hq, n_tokens]) in fp64.

    khat, vhat: [n_kv * n_tokens, 128] decoded K and V (any float dtype);
    q_bits: [B, Hq, 128] bf16 bit patterns."""
    if Hq % n_kv != 0:
        raise ValueError("Hq must be a multiple of n_kv")
    G = Hq // n_kv
    K = np.asarray(khat, dtype=np.float64).reshape(n_kv, n_tokens, 128)
    V = np.asarray(vhat, dtype=np.float64).reshape(n_kv, n_tokens, 128)
    q = bf16_bits_to_f64(q_bits).reshape(B, Hq, 128)
    out = np.zeros((B, Hq, 128))
    P = np.zeros((B, Hq, n_tokens))
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            s = (K[h] @ q[b, hq]) * scale
            w = np.exp(s - s.max())
            p = w / w.sum()
            P[b, hq] = p
            out[b, hq] = p @ V[h]
    return out, P

"""Seeded synthetic inputs shaped like the workloads the HyperQuant summary
evaluates on (Llama-3.1-8B KV cache and linear weights; "Experimental
results" section).  No trained weights or datasets are used: tensors of the
same shapes and value distributions stand in for them.

This module holds no arithmetic of the codec itself (no transform, lattice,
dither or sign mask): it only draws data, so that the CUDA path and the CPU
oracle can be fed identical tensors.  Data drawn on CPU and on CUDA differ
(different generator engines); a comparison always feeds both sides the same
tensor.

Recipes (seeds are fixed; bf16 values are fp32 draws rounded to nearest even):
  tiny KV      [256, 128]  N(0, 1); exactly 1% of coordinates (328), picked
               without replacement, scaled x20.
  KV cache     [layers][K,V][8 heads][tokens][128]  Student-t (nu = 5) times a
               lognormal(0, 1) scale per (layer, K/V, head, channel), with 4
               random outlier channels per (layer, K/V, head) scaled x10.
  weights      [out][in]  N(0, 0.02^2), Bernoulli(0.001) entries x15; tiles of
               128 run along the input dimension (row-major order).
  queries      [batch][q heads][128]  N(0, 1).
"""
from __future__ import annotations

import torch

TILE = 128

# Fixed seeds of the five workloads (data seed, then codec seeds).
TINY = dict(data_seed=0, sign_seed=0, dither_seed=0, n_tokens=256)
KV8B = dict(data_seed=2, sign_seed=20, layer_sign_seed=21, dither_seed=22,
            layers=32, kv_heads=8, tokens=8192)
WEIGHTS8B = dict(data_seed=3, sign_seed=30,
                 shapes=((4096, 4096), (1024, 4096), (4096, 14336), (14336, 4096)))
LONGCTX = dict(data_seed=4, sign_seed=40, layer_sign_seed=41, dither_seed=42,
               kv_heads=8, tokens=131072)
SCORES = dict(data_seed=5, sign_seed=50, layer_sign_seed=51, kv_heads=8, tokens=32768,
              batch=16, q_heads=32, q_seed=55, dither_seeds=tuple(range(500, 564)))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def tiny_kv(device="cpu") -> torch.Tensor:
    """[256, 128] bf16: N(0,1) with 328 coordinates x20."""
    g = _gen(TINY["data_seed"], device)
    n = TINY["n_tokens"] * TILE
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    idx = torch.randperm(n, generator=g, device=device)[: round(0.01 * n)]   # 328 of 32768
    x[idx] *= 20.0
    return x.to(torch.bfloat16).reshape(TINY["n_tokens"], TILE)


def kv_scales(seed: int, kv_heads: int) -> torch.Tensor:
    """Per-channel scales [kv_heads, 1, 128] of one slab: lognormal(0, 1), with 4
    random outlier channels per head x10.  Always drawn on the CPU, so a slab
    drawn on any device has the same scales (only the bulk noise differs)."""
    g = _gen(seed, "cpu")
    scale = torch.exp(torch.randn((kv_heads, 1, TILE), generator=g))
    for h in range(kv_heads):
        ch = torch.randperm(TILE, generator=g)[:4]
        scale[h, 0, ch] *= 10.0
    return scale


def kv_slab(seed: int, kv_heads: int, tokens: int, device="cpu") -> torch.Tensor:
    """One (layer, K-or-V) slab [kv_heads, tokens, 128] bf16: Student-t (nu = 5)
    noise times the slab's per-channel scales."""
    g = _gen(seed + 7919, device)
    shape = (kv_heads, tokens, TILE)
    num = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(5):
        n = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(n, n)
    t = num / torch.sqrt(chi2 / 5.0)
    del chi2, num
    return (t * kv_scales(seed, kv_heads).to(device)).to(torch.bfloat16)


def slab_seed(data_seed: int, layer: int, kv: int) -> int:
    return data_seed * 100003 + layer * 2 + kv


def kv_cache_8b(device="cuda", layers: int | None = None, tokens: int | None = None) -> torch.Tensor:
    """Llama-3.1-8B-shaped KV cache [layers, 2, 8, tokens, 128] bf16."""
    L = KV8B["layers"] if layers is None else layers
    T = KV8B["tokens"] if tokens is None else tokens
    out = torch.empty((L, 2, KV8B["kv_heads"], T, TILE), dtype=torch.bfloat16, device=device)
    for l in range(L):
        for kv in range(2):
            out[l, kv] = kv_slab(slab_seed(KV8B["data_seed"], l, kv), KV8B["kv_heads"], T, device)
    return out


def long_context_layer(device="cuda", tokens: int | None = None) -> torch.Tensor:
    """One layer's K and V [2, 8, tokens, 128] bf16 (KV-cache distribution)."""
    T = LONGCTX["tokens"] if tokens is None else tokens
    out = torch.empty((2, LONGCTX["kv_heads"], T, TILE), dtype=torch.bfloat16, device=device)
    for kv in range(2):
        out[kv] = kv_slab(slab_seed(LONGCTX["data_seed"], 0, kv), LONGCTX["kv_heads"], T, device)
    return out


def scores_keys(device="cuda", tokens: int | None = None) -> torch.Tensor:
    """K [8, tokens, 128] bf16 for the fused-scores workload."""
    T = SCORES["tokens"] if tokens is None else tokens
    return kv_slab(slab_seed(SCORES["data_seed"], 0, 0), SCORES["kv_heads"], T, device)


def scores_values(device="cuda", tokens: int | None = None) -> torch.Tensor:
    """V [8, tokens, 128] bf16 for the decode-attention workload (the V slab of
    the same layer as scores_keys)."""
    T = SCORES["tokens"] if tokens is None else tokens
    return kv_slab(slab_seed(SCORES["data_seed"], 0, 1), SCORES["kv_heads"], T, device)


def scores_queries(device="cuda", batch: int | None = None, q_heads: int | None = None) -> torch.Tensor:
    """q [batch, q_heads, 128] bf16, N(0, 1)."""
    B = SCORES["batch"] if batch is None else batch
    H = SCORES["q_heads"] if q_heads is None else q_heads
    g = _gen(SCORES["q_seed"], device)
    return torch.randn((B, H, TILE), generator=g, device=device).to(torch.bfloat16)


def haar_rotations(n: int, seed: int = 88):
    """[n][128][128] fp32 numpy: n independent Haar-uniform orthogonal
    matrices (QR of a Gaussian matrix with the signs of R's diagonal moved
    into Q), drawn on the CPU so that every device gets the same values."""
    import numpy as np
    g = _gen(seed, "cpu")
    a = torch.randn((n, TILE, TILE), generator=g, dtype=torch.float64)
    q, r = torch.linalg.qr(a)
    q = q * torch.sign(torch.diagonal(r, dim1=-2, dim2=-1)).unsqueeze(-2)
    return np.ascontiguousarray(q.to(torch.float32).numpy())


def activations(batch: int, cols: int, seed: int = 77, device="cuda") -> torch.Tensor:
    """x [batch, cols] bf16, N(0, 1): the activations multiplied by a weight matrix."""
    g = _gen(seed, device)
    return torch.randn((batch, cols), generator=g, device=device).to(torch.bfloat16)


def weight_matrix(index: int, device="cuda", rows: int | None = None) -> torch.Tensor:
    """Llama-3.1-8B-shaped linear weight [out, in] bf16 (optionally the first `rows` rows)."""
    out_f, in_f = WEIGHTS8B["shapes"][index]
    R = out_f if rows is None else rows
    g = _gen(WEIGHTS8B["data_seed"] * 1000 + index, device)
    w = torch.randn((R, in_f), generator=g, device=device) * 0.02
    hit = torch.rand((R, in_f), generator=g, device=device) < 0.001
    w = torch.where(hit, w * 15.0, w)
    return w.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (on the host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")

"""Shared helpers of the GPU parity tests: run one case through the CUDA
library (C ABI via the binding) and through the CPU oracle on the same
tensors, and compare."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CAL = os.path.join(ROOT, "weights_hq_encode_gb300", "calibration.json")


def calibration():
    with open(CAL) as f:
        return json.load(f)


def bits_to_torch(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).to(device)


class Case:
    """One codec configuration with its inputs on both sides."""

    def __init__(self, x_bits: np.ndarray, lattice: int, k: int, alpha: float, dither: int,
                 seed: int, masks: np.ndarray, tps: int, tile_base: int = 0, rot=None):
        self.x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1, 128)
        self.n = self.x_bits.shape[0]
        self.lattice, self.k, self.alpha, self.dither, self.seed = lattice, k, alpha, dither, seed
        self.masks = np.ascontiguousarray(masks, dtype=np.uint32).reshape(-1, 4)
        self.tps, self.tile_base = tps, tile_base
        self.rot = None if rot is None else np.ascontiguousarray(rot, dtype=np.float32)

    def oracle_params(self, O):
        return O.make_params(self.lattice, self.k, self.alpha, self.dither, self.seed, self.masks,
                             self.tps, self.tile_base, rot=self.rot)

    def gpu_params(self, hq, **kw):
        signs = torch.from_numpy(self.masks.view(np.int32).copy()).cuda()
        rot = None if self.rot is None else torch.from_numpy(self.rot.copy()).cuda()
        return hq.make_params(self.lattice, self.k, self.alpha, self.dither, self.seed, signs,
                              self.tps, self.tile_base, rot=rot, **kw)


def gpu_encode(hq, p, x: torch.Tensor, n: int, cap=None):
    """Size query + encode through the C ABI; returns (stream, offsets, status, total)."""
    dev = x.device
    offsets = torch.zeros(hq.hq_num_groups(n) + 1, dtype=torch.int64, device=dev)
    ws = torch.zeros(max(hq.hq_encode_workspace_bytes(n), 8), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = hq.hq_encode(p, x, n, None, 0, offsets, ws, status)
    assert rc == hq.HQ_OK, rc
    total = int(offsets[-1].item()) if n > 0 else 0
    if cap is None:
        cap = total
    stream = torch.full((max(cap, 1) + 8,), -1, dtype=torch.int32, device=dev)   # guard words
    st_size = int(status.item())
    status.zero_()
    rc = hq.hq_encode(p, x, n, stream, cap, offsets, ws, status)
    assert rc == hq.HQ_OK, rc
    torch.cuda.synchronize()
    return stream, offsets, int(status.item()), total, st_size


def gpu_decode(hq, p, stream, words, offsets, n, kind):
    dt = torch.float32 if kind == hq.HQ_OUT_F32 else torch.bfloat16
    out = torch.full((max(n, 1), 128), 7.0, dtype=dt, device=stream.device)
    status = torch.zeros(1, dtype=torch.int32, device=stream.device)
    rc = hq.hq_decode(p, stream, words, offsets, n, out, kind, status)
    assert rc == hq.HQ_OK, rc
    torch.cuda.synchronize()
    return out[:n], int(status.item())


def u32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)

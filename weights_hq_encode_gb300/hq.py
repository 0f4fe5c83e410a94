"""Thin Python binding of the C ABI in ``include/hq.h`` (argument marshalling only).

Every entry point of the library has a function of the same name here that
takes torch tensors (device memory and streams come from PyTorch) and passes
raw pointers through ctypes.  All of the codec's work happens in the CUDA
kernels of ``_build/libhq.so``; there is no CPU fallback: importing this
module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

HQ_OK, HQ_ERR_INVALID, HQ_ERR_CUDA, HQ_ERR_CAPACITY = 0, 1, 2, 4
HQ_ERR_CORRUPT, HQ_ERR_TIMEOUT, HQ_ERR_RANGE = 8, 16, 32
HQ_Z, HQ_A2, HQ_D4, HQ_E8 = 1, 2, 4, 8
HQ_OUT_BF16, HQ_OUT_F32 = 0, 1
HQ_TILE, HQ_GROUP_TILES = 128, 32
HQ_FLAG_WORKSPACE_READY = 1

EXPORTED = ("hq_num_groups", "hq_encode_workspace_bytes", "hq_encode", "hq_decode",
            "hq_decode_qk_workspace_bytes", "hq_decode_qk", "hq_make_signs",
            "hq_make_layer_signs", "hq_status_string",
            "hq_encode_noalloc", "hq_payload_bits", "hq_calibrate",
            "hq_decode_attention_workspace_bytes", "hq_decode_attention",
            "hq_decode_gemm_workspace_bytes", "hq_decode_gemm")
HQ_NOALLOC_MAX_TILES = 1 << 22


class hq_params(ctypes.Structure):
    _fields_ = [("lattice", ctypes.c_int32), ("rice_k", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("dither", ctypes.c_int32),
                ("dither_seed", ctypes.c_uint64), ("tile_base", ctypes.c_uint64),
                ("d_signs", ctypes.c_void_p), ("tiles_per_segment", ctypes.c_int64),
                ("lookback_spins", ctypes.c_uint32), ("flags", ctypes.c_uint32),
                ("d_rot", ctypes.c_void_p)]


class hq_calibration(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("rice_k", ctypes.c_int32), ("bps", ctypes.c_double),
                ("feasible", ctypes.c_int32), ("evaluations", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} (run weights_hq_encode_gb300.build)")
    L = ctypes.CDLL(path)
    vp, i64, u64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    L.hq_num_groups.restype = i64
    L.hq_num_groups.argtypes = [i64]
    L.hq_encode_workspace_bytes.restype = sz
    L.hq_encode_workspace_bytes.argtypes = [i64]
    L.hq_encode.restype = ctypes.c_int
    L.hq_encode.argtypes = [vp, vp, i64, vp, u64, vp, vp, sz, vp, vp]
    L.hq_encode_noalloc.restype = ctypes.c_int
    L.hq_encode_noalloc.argtypes = [vp, vp, i64, vp, u64, vp, vp, vp]
    L.hq_payload_bits.restype = ctypes.c_int
    L.hq_payload_bits.argtypes = [vp, vp, i64, vp, vp, sz, vp, vp]
    L.hq_calibrate.restype = ctypes.c_int
    L.hq_calibrate.argtypes = [vp, vp, i64, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                               ctypes.c_int, vp, sz, vp, vp, vp, vp]
    L.hq_decode.restype = ctypes.c_int
    L.hq_decode.argtypes = [vp, vp, u64, vp, i64, vp, ctypes.c_int, vp, vp]
    L.hq_decode_qk_workspace_bytes.restype = sz
    L.hq_decode_qk_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    L.hq_decode_qk.restype = ctypes.c_int
    L.hq_decode_qk.argtypes = [vp, vp, u64, vp, ctypes.c_int, i64, vp, ctypes.c_int,
                               ctypes.c_int, vp, vp, sz, vp, vp]
    L.hq_decode_attention_workspace_bytes.restype = sz
    L.hq_decode_attention_workspace_bytes.argtypes = [ctypes.c_int, i64, ctypes.c_int, ctypes.c_int]
    L.hq_decode_attention.restype = ctypes.c_int
    L.hq_decode_attention.argtypes = [vp, vp, u64, vp, vp, vp, u64, vp, ctypes.c_int, i64, vp,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_float, vp, vp, vp, sz,
                                      vp, vp]
    L.hq_decode_gemm_workspace_bytes.restype = sz
    L.hq_decode_gemm_workspace_bytes.argtypes = [i64, i64, ctypes.c_int]
    L.hq_decode_gemm.restype = ctypes.c_int
    L.hq_decode_gemm.argtypes = [vp, vp, u64, vp, i64, i64, vp, ctypes.c_int, vp, vp, sz, vp, vp]
    L.hq_make_signs.restype = None
    L.hq_make_signs.argtypes = [u64, u64, vp]
    L.hq_make_layer_signs.restype = None
    L.hq_make_layer_signs.argtypes = [u64, u64, u64, vp]
    L.hq_status_string.restype = ctypes.c_char_p
    L.hq_status_string.argtypes = [ctypes.c_int]
    return L


_lib = _load()


def lib():
    return _lib


# ------------------------------------------------------------------ marshalling
def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, name: str):
    if rc != HQ_OK:
        raise RuntimeError(f"{name}: {hq_status_string(rc)} ({rc})")


def make_params(lattice, rice_k, alpha, dither, dither_seed, signs: torch.Tensor,
                tiles_per_segment, tile_base=0, lookback_spins=0, flags=0,
                rot: torch.Tensor | None = None) -> hq_params:
    """hq_params with d_signs pointing at a device uint32 tensor [n_segments, 4]
    and, optionally, d_rot at a device fp32 tensor [n_segments, 128, 128]."""
    if signs.dtype not in (torch.int32, torch.uint32) or not signs.is_cuda:
        raise TypeError("signs must be a CUDA int32/uint32 tensor [n_segments, 4]")
    if rot is not None and (rot.dtype != torch.float32 or not rot.is_cuda or
                            not rot.is_contiguous()):
        raise TypeError("rot must be a contiguous CUDA fp32 tensor [n_segments, 128, 128]")
    p = hq_params(int(lattice), int(rice_k), float(alpha), int(dither), int(dither_seed),
                  int(tile_base), signs.data_ptr(), int(tiles_per_segment), int(lookback_spins),
                  int(flags), rot.data_ptr() if rot is not None else None)
    p._signs, p._rot = signs, rot      # keep the arrays alive as long as the params
    return p


# ------------------------------------------------------------------ same names as the C ABI
def hq_num_groups(n_tiles: int) -> int:
    return int(_lib.hq_num_groups(n_tiles))


def hq_encode_workspace_bytes(n_tiles: int) -> int:
    return int(_lib.hq_encode_workspace_bytes(n_tiles))


def hq_decode_qk_workspace_bytes(B: int, Hq: int) -> int:
    return int(_lib.hq_decode_qk_workspace_bytes(B, Hq))


def hq_encode(p: hq_params, x: torch.Tensor, n_tiles: int, stream_buf, cap_words: int,
              offsets: torch.Tensor, ws: torch.Tensor, status: torch.Tensor, stream=None) -> int:
    return int(_lib.hq_encode(ctypes.byref(p), _ptr(x), n_tiles, _ptr(stream_buf), cap_words,
                              _ptr(offsets), _ptr(ws), ws.numel() * ws.element_size(),
                              _ptr(status), _stream(stream)))


def hq_encode_noalloc(p: hq_params, x: torch.Tensor, n_tiles: int, stream_buf, cap_words: int,
                      offsets: torch.Tensor, status: torch.Tensor, stream=None) -> int:
    """hq_encode with the library's built-in scratch (no workspace argument)."""
    return int(_lib.hq_encode_noalloc(ctypes.byref(p), _ptr(x), n_tiles, _ptr(stream_buf),
                                      cap_words, _ptr(offsets), _ptr(status), _stream(stream)))


def hq_payload_bits(p: hq_params, x: torch.Tensor, n_tiles: int, bits: torch.Tensor,
                    ws: torch.Tensor, status: torch.Tensor, stream=None) -> int:
    """Adds the Rice payload bits of encoding x to the device int64 `bits`."""
    return int(_lib.hq_payload_bits(ctypes.byref(p), _ptr(x), n_tiles, _ptr(bits), _ptr(ws),
                                    ws.numel() * ws.element_size(), _ptr(status),
                                    _stream(stream)))


def hq_calibrate(p: hq_params, x: torch.Tensor, n_tiles: int, target_bps: float, tol: float,
                 k_min: int, k_max: int, ws: torch.Tensor, bits: torch.Tensor,
                 status: torch.Tensor, stream=None):
    """(return code, hq_calibration) of the GPU rate calibration."""
    out = hq_calibration()
    rc = int(_lib.hq_calibrate(ctypes.byref(p), _ptr(x), n_tiles, float(target_bps), float(tol),
                               k_min, k_max, _ptr(ws), ws.numel() * ws.element_size(), _ptr(bits),
                               _ptr(status), _stream(stream), ctypes.byref(out)))
    return rc, out


def hq_decode(p: hq_params, stream_buf: torch.Tensor, stream_words: int, offsets: torch.Tensor,
              n_tiles: int, out: torch.Tensor, out_kind: int, status: torch.Tensor,
              stream=None) -> int:
    return int(_lib.hq_decode(ctypes.byref(p), _ptr(stream_buf), stream_words, _ptr(offsets),
                              n_tiles, _ptr(out), out_kind, _ptr(status), _stream(stream)))


def hq_decode_qk(p: hq_params, k_stream: torch.Tensor, stream_words: int, k_offsets: torch.Tensor,
                 n_kv_heads: int, n_tokens: int, q: torch.Tensor, B: int, Hq: int,
                 scores: torch.Tensor, ws: torch.Tensor, status: torch.Tensor, stream=None) -> int:
    return int(_lib.hq_decode_qk(ctypes.byref(p), _ptr(k_stream), stream_words, _ptr(k_offsets),
                                 n_kv_heads, n_tokens, _ptr(q), B, Hq, _ptr(scores), _ptr(ws),
                                 ws.numel() * ws.element_size(), _ptr(status), _stream(stream)))


def hq_decode_attention_workspace_bytes(n_kv_heads: int, n_tokens: int, B: int, Hq: int) -> int:
    return int(_lib.hq_decode_attention_workspace_bytes(n_kv_heads, n_tokens, B, Hq))


def hq_decode_attention(pk: hq_params, k_stream: torch.Tensor, k_words: int,
                        k_offsets: torch.Tensor, pv: hq_params, v_stream: torch.Tensor,
                        v_words: int, v_offsets: torch.Tensor, n_kv_heads: int, n_tokens: int,
                        q: torch.Tensor, B: int, Hq: int, scale: float, out: torch.Tensor,
                        probs, ws: torch.Tensor, status: torch.Tensor, stream=None) -> int:
    return int(_lib.hq_decode_attention(
        ctypes.byref(pk), _ptr(k_stream), k_words, _ptr(k_offsets), ctypes.byref(pv),
        _ptr(v_stream), v_words, _ptr(v_offsets), n_kv_heads, n_tokens, _ptr(q), B, Hq,
        float(scale), _ptr(out), _ptr(probs), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(status), _stream(stream)))


def hq_decode_gemm_workspace_bytes(rows: int, cols: int, B: int) -> int:
    return int(_lib.hq_decode_gemm_workspace_bytes(rows, cols, B))


def hq_decode_gemm(p: hq_params, w_stream: torch.Tensor, w_words: int, w_offsets: torch.Tensor,
                   rows: int, cols: int, x: torch.Tensor, B: int, y: torch.Tensor,
                   ws: torch.Tensor, status: torch.Tensor, stream=None) -> int:
    return int(_lib.hq_decode_gemm(ctypes.byref(p), _ptr(w_stream), w_words, _ptr(w_offsets),
                                   rows, cols, _ptr(x), B, _ptr(y), _ptr(ws),
                                   ws.numel() * ws.element_size(), _ptr(status),
                                   _stream(stream)))


def hq_make_signs(seed: int, segment: int):
    out = (ctypes.c_uint32 * 4)()
    _lib.hq_make_signs(seed, segment, out)
    return [int(v) for v in out]


def hq_make_layer_signs(seed_d: int, seed_s: int, layer: int):
    out = (ctypes.c_uint32 * 4)()
    _lib.hq_make_layer_signs(seed_d, seed_s, layer, out)
    return [int(v) for v in out]


def hq_status_string(status: int) -> str:
    return _lib.hq_status_string(int(status)).decode()


# ------------------------------------------------------------------ conveniences
def signs_tensor(masks, device="cuda") -> torch.Tensor:
    """[n_segments][4] masks (lists of 4 uint32) -> device int32 tensor."""
    import numpy as np
    a = np.asarray(masks, dtype=np.uint32).reshape(-1, 4).view(np.int32)
    return torch.from_numpy(a.copy()).to(device)


def kv_layer_masks(seed_d: int, seed_s: int, layers: int):
    """Per-layer masks D XOR S_layer (Method 1 and 4: two sign diagonals)."""
    return [hq_make_layer_signs(seed_d, seed_s, l) for l in range(layers)]


def as_tiles(x: torch.Tensor) -> torch.Tensor:
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.numel() % HQ_TILE:
        raise TypeError("expected a CUDA bf16 tensor with a multiple of 128 elements")
    return x.contiguous().view(-1, HQ_TILE).view(torch.int16)


class Encoded:
    """A stream, its group index and the params that produced it."""

    def __init__(self, stream, offsets, n_tiles, params, total_words):
        self.stream, self.offsets, self.n_tiles = stream, offsets, n_tiles
        self.params, self.total_words = params, total_words

    def nbytes(self) -> int:
        return self.total_words * 4 + self.offsets.numel() * 8


def encode(x: torch.Tensor, p: hq_params, stream=None) -> Encoded:
    """Size query, then encode (two launches; synchronises once to size the buffer)."""
    xt = as_tiles(x)
    n = xt.shape[0]
    dev = x.device
    offsets = torch.zeros(hq_num_groups(n) + 1, dtype=torch.int64, device=dev)
    ws = torch.empty(max(hq_encode_workspace_bytes(n), 8), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(hq_encode(p, xt, n, None, 0, offsets, ws, status, stream), "hq_encode(size)")
    total = int(offsets[-1].item())
    buf = torch.empty(max(total, 1), dtype=torch.int32, device=dev)
    status.zero_()
    _check(hq_encode(p, xt, n, buf, total, offsets, ws, status, stream), "hq_encode")
    st = int(status.item())
    if st & ~HQ_ERR_RANGE:
        raise RuntimeError(f"hq_encode: {hq_status_string(st)} ({st})")
    return Encoded(buf, offsets, n, p, total)


def decode(enc: Encoded, out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    kind = HQ_OUT_BF16 if out_dtype == torch.bfloat16 else HQ_OUT_F32
    out = torch.empty((enc.n_tiles, HQ_TILE), dtype=out_dtype, device=enc.stream.device)
    status = torch.zeros(1, dtype=torch.int32, device=enc.stream.device)
    _check(hq_decode(enc.params, enc.stream, enc.total_words, enc.offsets, enc.n_tiles, out, kind,
                     status, stream), "hq_decode")
    st = int(status.item())
    if st:
        raise RuntimeError(f"hq_decode: {hq_status_string(st)} ({st})")
    return out

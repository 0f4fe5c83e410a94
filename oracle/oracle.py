"""ctypes front end of the CPU oracle (``hq_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``.  The product library never
imports, links or calls anything here, and this module imports nothing from
the product package.

The C source is compiled on first use with the host compiler (gcc, ``-O2
-ffp-contract=off``, no fast-math) into ``oracle/_build/``.  With the
environment variable ``HQ_ORACLE_SRC`` set to another C file (a copy of
``hq_oracle.c`` with a mistake planted by ``tests/oracle_mutations.py``),
that file is compiled instead, into a library beside it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ALT = os.environ.get("HQ_ORACLE_SRC")
_SRC = os.path.abspath(_ALT) if _ALT else os.path.join(_HERE, "hq_oracle.c")
_BUILD = os.path.dirname(_SRC) if _ALT else os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libhq_oracle.so")
_lock = threading.Lock()
_lib = None

Z, A2, D4, E8 = 1, 2, 4, 8
OK, ERR_INVALID, ERR_CAPACITY, ERR_CORRUPT, ERR_RANGE = 0, 1, 4, 8, 32
TILE = 128


def build(force: bool = False) -> str:
    """Compile the oracle shared library; returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Params(ctypes.Structure):
    _fields_ = [("lattice", ctypes.c_int32), ("rice_k", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("dither", ctypes.c_int32),
                ("dither_seed", ctypes.c_uint64), ("tile_base", ctypes.c_uint64),
                ("signs", ctypes.c_void_p), ("tiles_per_segment", ctypes.c_int64),
                ("rot", ctypes.c_void_p)]


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
            L.oracle_encode.restype = i64
            L.oracle_encode.argtypes = [vp, vp, i64, vp, u64, vp, vp, vp, vp, ctypes.c_int]
            L.oracle_payload_bits.restype = i64
            L.oracle_payload_bits.argtypes = [vp, vp, i64, ctypes.c_int]
            L.oracle_decode.restype = ctypes.c_int
            L.oracle_decode.argtypes = [vp, vp, u64, vp, i64, vp, vp, vp, vp, ctypes.c_int]
            L.oracle_scores.restype = ctypes.c_int
            L.oracle_scores.argtypes = [vp, ctypes.c_int, i64, vp, ctypes.c_int, ctypes.c_int,
                                        vp, ctypes.c_int]
            L.oracle_make_signs.argtypes = [u64, u64, vp]
            L.oracle_philox4x32_10.argtypes = [vp, vp, vp]
            L.oracle_fwht128.argtypes = [vp]
            L.oracle_nearest_e8.argtypes = [vp, vp]
            L.oracle_nearest_d4.argtypes = [vp, vp]
            L.oracle_nearest_a2.argtypes = [vp, vp]
            L.oracle_point.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int]
            L.oracle_nearest_z.restype = ctypes.c_int32
            L.oracle_nearest_z.argtypes = [ctypes.c_float]
            L.oracle_dither.argtypes = [ctypes.c_int, u64, u64, vp]
            L.oracle_fold.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int]
            L.oracle_rotate.argtypes = [vp, vp, vp]
            L.oracle_rotate_t.argtypes = [vp, vp, vp]
            L.oracle_unfold.restype = ctypes.c_int
            L.oracle_unfold.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_int]
            L.oracle_bit_stripped.restype = ctypes.c_int
            L.oracle_bit_stripped.argtypes = [ctypes.c_int] * 4
            L.oracle_tile_rbits.restype = i64
            L.oracle_tile_rbits.argtypes = [ctypes.c_int, ctypes.c_int]
            L.oracle_n_groups.restype = i64
            L.oracle_n_groups.argtypes = [i64]
            L.oracle_encode_scale.restype = ctypes.c_float
            L.oracle_encode_scale.argtypes = [ctypes.c_float]
            L.oracle_decode_scale.restype = ctypes.c_float
            L.oracle_decode_scale.argtypes = [ctypes.c_float]
            L.oracle_e8_rule_census.restype = ctypes.c_int
            L.oracle_e8_rule_census.argtypes = [vp, vp, i64, vp, vp, ctypes.c_int]
            L.oracle_scale_rounding_census.restype = ctypes.c_int
            L.oracle_scale_rounding_census.argtypes = [vp, vp, i64, vp, vp, ctypes.c_int]
            L.oracle_e8_plain.argtypes = [vp, vp]
            L.oracle_group_tiles.restype = ctypes.c_int
            L.oracle_range_limit.restype = ctypes.c_float
            L.oracle_symbol_limit.restype = ctypes.c_uint32
            _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ----------------------------------------------------------------- primitives
def philox(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def make_signs(seed: int, segment: int) -> np.ndarray:
    out = np.zeros(4, np.uint32)
    lib().oracle_make_signs(seed, segment, _p(out))
    return out


def fwht128(x) -> np.ndarray:
    a = np.array(x, dtype=np.float32, copy=True).reshape(128)
    lib().oracle_fwht128(_p(a))
    return a


def nearest_e8(y) -> np.ndarray:
    a = np.ascontiguousarray(y, dtype=np.float32).reshape(8)
    v = np.zeros(8, np.int32)
    lib().oracle_nearest_e8(_p(a), _p(v))
    return v


def nearest_d4(y) -> np.ndarray:
    a = np.ascontiguousarray(y, dtype=np.float32).reshape(4)
    v = np.zeros(4, np.int32)
    lib().oracle_nearest_d4(_p(a), _p(v))
    return v


def nearest_a2(y) -> np.ndarray:
    """Codes (m, n) of the nearest A2 point to y (2 floats)."""
    a = np.ascontiguousarray(y, dtype=np.float32).reshape(2)
    v = np.zeros(2, np.int32)
    lib().oracle_nearest_a2(_p(a), _p(v))
    return v


def point(lattice: int, v) -> np.ndarray:
    """Lattice point (fp32 coordinates) of a code vector."""
    a = np.ascontiguousarray(v, dtype=np.int32)
    pt = np.zeros(a.size, np.float32)
    lib().oracle_point(lattice, _p(a), _p(pt), a.size)
    return pt


def rotate(R, x, transpose=False) -> np.ndarray:
    """R x (or R^T x) as the codec's fixed-order fp32 FMA chains."""
    Rm = np.ascontiguousarray(R, dtype=np.float32).reshape(128, 128)
    xv = np.ascontiguousarray(x, dtype=np.float32).reshape(128)
    out = np.zeros(128, np.float32)
    (lib().oracle_rotate_t if transpose else lib().oracle_rotate)(_p(Rm), _p(xv), _p(out))
    return out


def nearest_z(y: float) -> int:
    return int(lib().oracle_nearest_z(float(y)))


def dither(lattice: int, seed: int, tile: int) -> np.ndarray:
    u = np.zeros(128, np.float32)
    lib().oracle_dither(lattice, seed, tile, _p(u))
    return u


def fold(lattice: int, v) -> np.ndarray:
    a = np.ascontiguousarray(v, dtype=np.int32)
    s = np.zeros(a.size, np.uint32)
    lib().oracle_fold(lattice, _p(a), _p(s), a.size)
    return s


def unfold(lattice: int, k: int, s):
    a = np.ascontiguousarray(s, dtype=np.uint32)
    v = np.zeros(a.size, np.int32)
    rc = lib().oracle_unfold(lattice, k, _p(a), _p(v), a.size)
    return v, rc


def bit_stripped(lattice: int, coord: int, bit: int, k: int) -> bool:
    return bool(lib().oracle_bit_stripped(lattice, coord, bit, k))


def tile_rbits(lattice: int, k: int) -> int:
    return int(lib().oracle_tile_rbits(lattice, k))


def n_groups(n_tiles: int) -> int:
    return int(lib().oracle_n_groups(n_tiles))


def encode_scale(alpha: float) -> float:
    return float(lib().oracle_encode_scale(alpha))


def decode_scale(alpha: float) -> float:
    return float(lib().oracle_decode_scale(alpha))


GROUP_TILES = 32


# ----------------------------------------------------------------- codec
def make_params(lattice, rice_k, alpha, dither, dither_seed, signs, tiles_per_segment,
                tile_base=0, rot=None):
    """rot: None, or [n_segments][128][128] fp32 row-major rotations R (the
    tile is coded as RHT(R x))."""
    signs = np.ascontiguousarray(signs, dtype=np.uint32).reshape(-1, 4)
    R = None if rot is None else np.ascontiguousarray(rot, dtype=np.float32).reshape(-1, 128, 128)
    P = Params(lattice, rice_k, alpha, dither, dither_seed, tile_base,
               ctypes.c_void_p(signs.ctypes.data), tiles_per_segment,
               ctypes.c_void_p(R.ctypes.data) if R is not None else ctypes.c_void_p(0))
    P._keep = (signs, R)     # keep the arrays alive with the struct
    return P


def encode(P: Params, x_bf16_bits: np.ndarray, cap_words: int | None = None,
           want_codes: bool = False, threads: int | None = None):
    """Encode bf16 tiles given as uint16 bit patterns [n_tiles, 128].

    Returns dict(stream, offsets, status, total_words, codes?, tile_bits)."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16).reshape(-1, 128)
    n = x.shape[0]
    ng = n_groups(n)
    off = np.zeros(ng + 1, np.uint64)
    st = np.zeros(1, np.uint32)
    tb = np.zeros(max(n, 1), np.uint64)
    th = threads or default_threads()
    L = lib()
    if cap_words is None:   # size pass, then the real pass
        total = L.oracle_encode(ctypes.byref(P), _p(x), n, None, 0, _p(off), _p(st), None,
                                None, th)
        if total < 0:
            raise ValueError("oracle_encode: invalid arguments")
        cap_words = int(total)
        st[0] = 0
    stream = np.zeros(max(cap_words, 1), np.uint32)
    codes = np.zeros((n, 128), np.int32) if want_codes else None
    total = L.oracle_encode(ctypes.byref(P), _p(x), n, _p(stream), cap_words, _p(off), _p(st),
                            _p(codes), _p(tb), th)
    if total < 0:
        raise ValueError("oracle_encode: invalid arguments")
    return dict(stream=stream[:cap_words], offsets=off, status=int(st[0]), total_words=int(total),
                codes=codes, tile_bits=tb[:n])


def payload_bits(P: Params, x_bf16_bits: np.ndarray, threads: int | None = None) -> int:
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16).reshape(-1, 128)
    r = lib().oracle_payload_bits(ctypes.byref(P), _p(x), x.shape[0], threads or default_threads())
    if r < 0:
        raise ValueError("oracle_payload_bits failed")
    return int(r)


def decode(P: Params, stream: np.ndarray, offsets: np.ndarray, n_tiles: int,
           out: str = "f32", want_codes: bool = False, threads: int | None = None):
    """Decode; returns dict(out, status, codes?)."""
    s = np.ascontiguousarray(stream, dtype=np.uint32)
    o = np.ascontiguousarray(offsets, dtype=np.uint64)
    f = np.zeros((n_tiles, 128), np.float32) if out == "f32" else None
    b = np.zeros((n_tiles, 128), np.uint16) if out == "bf16" else None
    codes = np.zeros((n_tiles, 128), np.int32) if want_codes else None
    st = np.zeros(1, np.uint32)
    rc = lib().oracle_decode(ctypes.byref(P), _p(s), s.size, _p(o), n_tiles, _p(f), _p(b), _p(codes),
                             _p(st), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_decode: invalid arguments")
    return dict(out=f if out == "f32" else b, status=int(st[0]), codes=codes)


def scores(khat: np.ndarray, n_kv_heads: int, n_tokens: int, q_bf16_bits: np.ndarray,
           B: int, Hq: int, threads: int | None = None) -> np.ndarray:
    k = np.ascontiguousarray(khat, dtype=np.float32)
    q = np.ascontiguousarray(q_bf16_bits, dtype=np.uint16)
    out = np.zeros((B, Hq, n_tokens), np.float32)
    rc = lib().oracle_scores(_p(k), n_kv_heads, n_tokens, _p(q), B, Hq, _p(out),
                             threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_scores: invalid arguments")
    return out


def e8_plain(y) -> np.ndarray:
    """The plain E8 rule: both cosets by the D_n decoder, fp32 squared
    distances summed left to right (diagnostic; the codec uses nearest_e8)."""
    yy = np.ascontiguousarray(y, dtype=np.float32).reshape(8)
    v = np.zeros(8, np.int32)
    lib().oracle_e8_plain(_p(yy), _p(v))
    return v


def scale_rounding_census(P: Params, x_bf16_bits: np.ndarray, threads: int | None = None) -> dict:
    """Counts, over every lattice vector the oracle codes from these tiles,
    where the scale and dither rounded once (the codec's reading) and rounded
    twice pick different points; dist_sum > 0 means the once-rounded points
    are nearer to the exact values in total (diagnostic)."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16).reshape(-1, 128)
    out = np.zeros(3, np.int64)
    dist = np.zeros(2, np.float64)
    if lib().oracle_scale_rounding_census(ctypes.byref(P), _p(x), x.shape[0], _p(out), _p(dist),
                                          threads or default_threads()) != 0:
        raise ValueError("oracle_scale_rounding_census: invalid arguments")
    return dict(vectors=int(out[0]), differ=int(out[1]), skipped_tiles=int(out[2]),
                dist_sum=float(dist[0]), dist_max=float(dist[1]))


def e8_rule_census(P: Params, x_bf16_bits: np.ndarray, threads: int | None = None) -> dict:
    """Counts, over every 8-vector the oracle codes from these tiles, where
    nearest_e8 (fp32 linear identity) and the plain rule disagree."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16).reshape(-1, 128)
    out = np.zeros(3, np.int64)
    dist = np.zeros(2, np.float64)
    if lib().oracle_e8_rule_census(ctypes.byref(P), _p(x), x.shape[0], _p(out), _p(dist),
                                   threads or default_threads()) != 0:
        raise ValueError("oracle_e8_rule_census: invalid arguments")
    return dict(vectors=int(out[0]), differ=int(out[1]), coset_differ=int(out[2]),
                dist_sum=float(dist[0]), dist_max=float(dist[1]))

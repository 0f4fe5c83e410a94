"""Rate calibration of alpha and the Rice parameter k, on the CPU oracle only.

HyperQuant summary, Method 2 (alpha is calibrated so that the codes fit) and
Method 3 (realized rate within about 0.01 bps of the target; k chosen per
bit rate).  Reading: for every k whose smallest reachable rate is below the
target, bisect log(alpha) until the realized payload rate (Rice bits per
element, index and padding excluded) is within 0.002 bps of the target; keep
the feasible k with the largest alpha (least distortion), ties to the smaller
k.  Subsets: the tiny KV set whole (k fixed at 2); the first 256 tokens of
every (layer, K/V) slab of the Llama-3.1-8B KV cache (all per-channel scales
of the cache, which are drawn identically on every device); the first 512
rows of each weight matrix; the first 16384 tokens of the long-context layer.

Writes ``weights_hq_encode_gb300/calibration.json``.  Run:
``python -m oracle.calibrate [--only NAME] [--lattices E8,A2]``.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import oracle as O  # noqa: E402
from weights_hq_encode_gb300 import inputs as I  # noqa: E402

OUT = os.path.join(ROOT, "weights_hq_encode_gb300", "calibration.json")
TOL = 0.002
LATTICES = {"E8": O.E8, "D4": O.D4, "A2": O.A2, "Z": O.Z}


def rate(x, lattice, k, alpha, dither, seed, signs, tps) -> float:
    P = O.make_params(lattice, k, alpha, dither, seed, signs, tps)
    return O.payload_bits(P, x) / x.size


def bisect_alpha(x, lattice, k, target, dither, seed, signs, tps):
    lo, hi = -14.0, 18.0                       # log2(alpha)
    r_lo = rate(x, lattice, k, 2.0 ** lo, dither, seed, signs, tps)
    if r_lo > target - TOL / 2:
        return None                            # k cannot go this low
    best = None
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        r = rate(x, lattice, k, 2.0 ** mid, dither, seed, signs, tps)
        if best is None or abs(r - target) < abs(best[1] - target):
            best = (mid, r)
        if abs(r - target) <= TOL:
            break
        if r < target:
            lo = mid
        else:
            hi = mid
    a = float(np.float32(2.0 ** best[0]))
    return dict(alpha=a, k=k, bps=rate(x, lattice, k, a, dither, seed, signs, tps))


def calibrate(x, lattice, target, dither, seed, signs, tps, ks=range(0, 9)):
    found = [c for c in (bisect_alpha(x, lattice, k, target, dither, seed, signs, tps) for k in ks)
             if c is not None and abs(c["bps"] - target) <= TOL]
    if not found:
        raise RuntimeError(f"no feasible k for target {target}")
    found.sort(key=lambda c: (-c["alpha"], c["k"]))
    return found[0]


def kv_masks(seed_d, seed_s, layer):
    return (O.make_signs(seed_d, 0) ^ O.make_signs(seed_s, layer)).reshape(1, 4)


def run(only=None, lattices=None):
    res = json.load(open(OUT)) if os.path.exists(OUT) else {}
    t0 = time.time()

    if only in (None, "tiny_kv"):
        x = I.bf16_bits(I.tiny_kv()).reshape(-1, 128)
        c = calibrate(x, O.E8, 3.0, 1, I.TINY["dither_seed"], O.make_signs(I.TINY["sign_seed"], 0),
                      1 << 40, ks=[2])
        res["tiny_kv"] = {"E8": {"3.0": c}}
        print("tiny_kv", c, f"{time.time() - t0:.0f}s", flush=True)

    if only in (None, "kv_cache_8b"):
        C = I.KV8B
        xs, ms = [], []
        for layer in range(C["layers"]):
            for kv in (0, 1):
                xs.append(I.bf16_bits(I.kv_slab(I.slab_seed(C["data_seed"], layer, kv),
                                                C["kv_heads"], 256)).reshape(-1, 128))
                ms.append(kv_masks(C["sign_seed"], C["layer_sign_seed"], layer))
        x = np.concatenate(xs)
        m = np.concatenate(ms)                 # one mask per slab subset
        tps = xs[0].shape[0]
        res["kv_cache_8b"] = {"E8": {}}
        for target in (2.0, 3.0):
            c = calibrate(x, O.E8, target, 1, C["dither_seed"], m, tps)
            res["kv_cache_8b"]["E8"][str(target)] = c
            print("kv_cache_8b", target, c, f"{time.time() - t0:.0f}s", flush=True)

    if only in (None, "weights_8b"):
        C = I.WEIGHTS8B
        m = O.make_signs(C["sign_seed"], 0).reshape(1, 4)
        res["weights_8b"] = {"E8": {}}
        for target in (3.0, 4.0, 5.0):
            per = []
            for i in range(len(C["shapes"])):
                x = I.bf16_bits(I.weight_matrix(i, device="cpu", rows=512)).reshape(-1, 128)
                per.append(calibrate(x, O.E8, target, 0, 0, m, 1 << 40))
            res["weights_8b"]["E8"][str(target)] = per
            print("weights_8b", target, per, f"{time.time() - t0:.0f}s", flush=True)

    if only in (None, "long_context"):
        C = I.LONGCTX
        x = np.concatenate([I.bf16_bits(I.kv_slab(I.slab_seed(C["data_seed"], 0, kv), C["kv_heads"],
                                                  16384)).reshape(-1, 128) for kv in (0, 1)])
        m = kv_masks(C["sign_seed"], C["layer_sign_seed"], 0)
        res.setdefault("long_context", {})
        for name, lat in LATTICES.items():
            if lattices and name not in lattices:
                continue
            res["long_context"][name] = {}
            for target in (1.7, 2.0, 2.5, 3.0):
                c = calibrate(x, lat, target, 1, C["dither_seed"], m, 1 << 40)
                res["long_context"][name][str(target)] = c
                print("long_context", name, target, c, f"{time.time() - t0:.0f}s", flush=True)

    res["_doc"] = ("alpha and Rice k per workload and target payload rate (bits per element), "
                   "frozen by oracle/calibrate.py from the CPU oracle; bps = realized payload "
                   "rate on the calibration subset.")
    with open(OUT, "w") as f:
        json.dump(res, f, indent=1, sort_keys=True)
    print("wrote", OUT)


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", default=None)
    ap.add_argument("--lattices", default=None, help="comma-separated subset for long_context")
    a = ap.parse_args()
    run(a.only, a.lattices.split(",") if a.lattices else None)

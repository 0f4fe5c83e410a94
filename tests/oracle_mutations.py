"""Mutation check of the oracle's pins (a developer tool, not collected by
pytest; about ten minutes on 16 cores).

Each entry plants one plausible mistake in a copy of ``oracle/hq_oracle.c``:
a wrong constant, index, sign, order or rounding in one step of the method
(HyperQuant summary, Method 1-4, and the fused-scores reading).  The copy is
compiled through ``HQ_ORACLE_SRC`` and the CPU suite (``-m "not gpu"``,
without ``test_abi.py``, whose host-side checks compare the oracle with the
CUDA library rather than with a fact outside both) runs against it; a
mistake is caught when some test fails.  The one expected
survivor is the FWHT's stage order, a reading that no fact outside the
oracle fixes (other orders give the same transform up to rounding).

Run: ``python tests/oracle_mutations.py [NAME ...]``.
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "hq_oracle.c")

# (name, text in hq_oracle.c, replacement)
MUTATIONS = [
    ("Philox multiplier", "(uint64_t)0xD2511F53u * c0", "(uint64_t)0xD2511F55u * c0"),
    ("Philox 9 rounds", "for (int round = 0; round < 10; ++round)",
     "for (int round = 0; round < 9; ++round)"),
    ("Philox key increment", "k0 += 0x9E3779B9u;", "k0 += 0x9E3779B1u;"),
    ("Philox word mix", "c2 = hi0 ^ c3 ^ k1;", "c2 = hi0 ^ c1 ^ k1;"),
    ("sign counter tag", "0x5349474Eu};", "0x5349474Fu};"),
    ("sign counter high word", "uint32_t ctr[4] = {(uint32_t)segment, (uint32_t)(segment >> 32), 0u,",
     "uint32_t ctr[4] = {(uint32_t)segment, 0u, 0u,"),
    ("FWHT stage order (a reading: expected to survive)",
     "for (int h = 1; h < TILE; h <<= 1) {\n    for (int i = 0; i < TILE; ++i) {\n      if (i & h) continue;",
     "for (int h = 64; h >= 1; h >>= 1) {\n    for (int i = 0; i < TILE; ++i) {\n      if (i & h) continue;"),
    ("FWHT difference sign", "x[i + h] = a - b;", "x[i + h] = b - a;"),
    ("Z ties away from zero", "return (int32_t)rintf(y);", "return (int32_t)roundf(y);"),
    ("dither grid points, not midpoints", "b[2 * m] = (float)(w[m] & 0xFFFFu) + 0.5f;",
     "b[2 * m] = (float)(w[m] & 0xFFFFu);"),
    ("dither high half", "b[2 * m + 1] = (float)(w[m] >> 16) + 0.5f;",
     "b[2 * m + 1] = (float)((w[m] >> 8) & 0xFFFFu) + 0.5f;"),
    ("dither counter j",
     "uint32_t ctr[4] = {(uint32_t)tile, (uint32_t)(tile >> 32), j, 0x44495448u};",
     "uint32_t ctr[4] = {(uint32_t)tile, (uint32_t)(tile >> 32), 15u - j, 0x44495448u};"),
    ("E8 dither box", "u0[7] = -2.0f + b[7] * 0x1p-14f;", "u0[7] = -1.0f + b[7] * 0x1p-15f;"),
    ("E8 dither not reduced", "for (int i = 0; i < 8; ++i) uj[i] = u0[i] - (float)lam[i];",
     "for (int i = 0; i < 8; ++i) uj[i] = u0[i];"),
    ("D4 dither box", "u0[3] = -1.0f + b[4 * h + 3] * 0x1p-15f;",
     "u0[3] = -0.5f + b[4 * h + 3] * 0x1p-16f;"),
    ("A2 dither box", "u0[1] = A2_H * (-1.0f + b[2 * h + 1] * 0x1p-15f);",
     "u0[1] = A2_H * (-0.5f + b[2 * h + 1] * 0x1p-16f);"),
    ("Z dither box", "for (int i = 0; i < 8; ++i) uj[i] = -0.5f + b[i] * 0x1p-16f;",
     "for (int i = 0; i < 8; ++i) uj[i] = -0.25f + b[i] * 0x1p-17f;"),
    ("dither ignores tile_base",
     "oracle_dither(P->lattice, P->dither_seed, P->tile_base + (uint64_t)t, u);\n  else for (int i = 0; i < TILE; ++i) u[i] = 0.0f;\n}",
     "oracle_dither(P->lattice, P->dither_seed, (uint64_t)t, u);\n  else for (int i = 0; i < TILE; ++i) u[i] = 0.0f;\n}"),
    ("E8 fold s_7", "s[b + 7] = 4u * zigzag(t) + 2u * (uint32_t)r + (uint32_t)p;",
     "s[b + 7] = 4u * zigzag(t) + (uint32_t)r + 2u * (uint32_t)p;"),
    ("E8 fold parity over 8", "for (int i = 0; i < 7; ++i) r += w[i];\n      r &= 1;\n      int32_t t",
     "for (int i = 0; i < 8; ++i) r += w[i];\n      r &= 1;\n      int32_t t"),
    ("D4 fold parity", "s[b + 3] = 2u * zigzag(t) + (uint32_t)r;",
     "s[b + 3] = 2u * zigzag(t) + (uint32_t)(1 - r);"),
    ("A2 fold sign", "s[b] = zigzag(v[b + 1]);", "s[b] = zigzag(-v[b + 1]);"),
    ("zigzag", "return n >= 0 ? 2u * (uint32_t)n : 2u * (uint32_t)(-(int64_t)n) - 1u;",
     "return n > 0 ? 2u * (uint32_t)n - 1u : 2u * (uint32_t)(-(int64_t)n);"),
    ("E8 unfold w_7", "w[7] = 2 * unzigzag(s[7] >> 2) + r;", "w[7] = 2 * unzigzag(s[7] >> 2) - r;"),
    ("E8 stripped bit", "if (bit == 1 && coord == 7) return 1;", "if (bit == 1 && coord == 6) return 1;"),
    ("encode scale", "return (float)((double)alpha / sqrt(128.0)); }",
     "return (float)((double)alpha / 128.0); }"),
    ("decode scale", "return (float)(1.0 / ((double)alpha * sqrt(128.0))); }",
     "return (float)(1.0 / ((double)alpha * 128.0)); }"),
    ("two roundings for scale and dither", "y[i] = fmaf(z[i], s, u[i]);", "y[i] = z[i] * s + u[i];"),
    ("encoder ignores the sign mask",
     "for (int i = 0; i < TILE; ++i) z[i] = mask_bit(m, i) ? -xf[i] : xf[i];",
     "for (int i = 0; i < TILE; ++i) z[i] = xf[i];"),
    ("decoder ignores the sign mask", "out[i] = mask_bit(m, i) ? -r : r;", "out[i] = r;"),
    ("mask bit order",
     "static int mask_bit(const uint32_t *m, int i) { return (int)((m[i >> 5] >> (i & 31)) & 1u); }",
     "static int mask_bit(const uint32_t *m, int i) { return (int)((m[i >> 5] >> (31 - (i & 31))) & 1u); }"),
    ("range limit", "if (!(fabsf(y[i]) <= RANGE_LIMIT)) flag = ORA_ERR_RANGE;",
     "if (!(fabsf(y[i]) < RANGE_LIMIT * 0.5f)) flag = ORA_ERR_RANGE;"),
    ("remainder bit order",
     "for (int bit = k - 1; bit >= 0; --bit)\n          if (!oracle_bit_stripped(C->P->lattice, j % dim, bit, k))\n            put_bit",
     "for (int bit = 0; bit < k; ++bit)\n          if (!oracle_bit_stripped(C->P->lattice, j % dim, bit, k))\n            put_bit"),
    ("LSB-first packing", "if (bit && w < cap) words[w] |= 0x80000000u >> (b & 31);",
     "if (bit && w < cap) words[w] |= 1u << (b & 31);"),
    ("A2 constant h", "static const float A2_H = 0.86602540378443865f;",
     "static const float A2_H = 0.8660254f + 1e-6f;"),
    ("rotation transposed", "oracle_rotate(tile_rot(P, t), xf, xf);", "oracle_rotate_t(tile_rot(P, t), xf, xf);"),
    ("GQA head map", "int h = hq / group;", "int h = hq % C->n_kv;"),
    ("decoder skips the FWHT", "  oracle_fwht128(z);\n  float s = oracle_decode_scale(P->alpha);",
     "  float s = oracle_decode_scale(P->alpha);"),
    ("unary length without terminator",
     "for (int j = 0; j < TILE; ++j) u += (uint64_t)(s[j] >> C->P->rice_k) + 1u;",
     "for (int j = 0; j < TILE; ++j) u += (uint64_t)(s[j] >> C->P->rice_k);"),
    ("decoder adds the dither", "for (int i = 0; i < TILE; ++i) z[i] = pt[i] - u[i];",
     "for (int i = 0; i < TILE; ++i) z[i] = pt[i] + u[i];"),
]


def run(names=None) -> int:
    orig = open(SRC).read()
    survived = []
    with tempfile.TemporaryDirectory(prefix="hq_oracle_mut_") as tmp:
        for name, old, new in MUTATIONS:
            if names and name not in names:
                continue
            if orig.count(old) != 1:
                print(f"{name}: pattern not found once in hq_oracle.c", flush=True)
                survived.append(name)
                continue
            d = os.path.join(tmp, str(len(os.listdir(tmp))))
            os.makedirs(d)
            alt = os.path.join(d, "hq_oracle.c")
            with open(alt, "w") as f:
                f.write(orig.replace(old, new))
            env = dict(os.environ, HQ_ORACLE_SRC=alt)
            r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-m", "not gpu", "-x", "-q",
                                "-p", "no:cacheprovider", "--ignore=tests/test_abi.py"], cwd=ROOT,
                               env=env, capture_output=True, text=True)
            failed = [l for l in r.stdout.splitlines() if l.startswith("FAILED")]
            if r.returncode != 0:
                print(f"caught    {name}: {failed[0] if failed else r.stdout.strip().splitlines()[-1]}",
                      flush=True)
            else:
                print(f"SURVIVED  {name}", flush=True)
                survived.append(name)
    print(f"{len(survived)} survived: {survived}")
    return 0


if __name__ == "__main__":
    sys.exit(run(sys.argv[1:] or None))

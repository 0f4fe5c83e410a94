/*
 * hq_oracle.c -- plain, slow CPU oracle for the HyperQuant tile codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that the tests, the smoke check and the CPU
 * baseline leg of the benchmark can check the CUDA library against an
 * independent statement of what the method computes.  It shares no code,
 * header, table or constant generator with the CUDA library.
 *
 * Sources (page titles and sections of the HyperQuant technical summaries):
 *   [RHT]    HyperQuant summary, Method 1 "Per-tile randomized Hadamard
 *            transform": tiles of 128, RHT_n(x) = H_n D x, H_n Walsh-Hadamard,
 *            D a random sign diagonal; the transform is orthogonal.
 *   [LAT]    Method 2 "Lattice quantization": E8 / D4 / Z, closed-form O(1)
 *            decoder for E8, integer embedding E8_int in Z^8, scale alpha.
 *   [STRIP]  Method 3 "Bit stripping and Rice coding": bits fixed by lattice
 *            membership (E8 parity) are removed losslessly; the remaining
 *            symbols are Rice coded with an unbounded codebook.
 *   [BIAS]   Method 4 "Bias correction for the KV cache": per-layer +-1 sign
 *            rotation; subtractive dither U ~ Uniform(V(Lambda)) added before
 *            quantization and subtracted after.
 *   [FUSED]  Significance / conclusion: fused decode + MMA as future work
 *            (here: attention scores q.K^T computed from compressed K).
 * Philox4x32-10 follows Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
 * as easy as 1, 2, 3" (SC'11).  Nearest-point rules follow Conway & Sloane,
 * "Fast quantizing and decoding algorithms for lattice quantizers" (1982).
 *
 * Where the summaries are silent the oracle takes one explicit reading; each
 * one is stated at the function that implements it.
 *
 * Arithmetic: IEEE binary32 with round-to-nearest-even.  Build with
 * -ffp-contract=off and without -ffast-math: every product and sum below is
 * rounded exactly where it is written, and fmaf() is used only where a fused
 * multiply-add is part of the definition.
 *
 * Parity status: every function here is pinned by a CPU test (known-answer
 * vectors, brute-force nearest point, exhaustive round trips, closed forms,
 * measured second moments, exact-arithmetic references); none is "parity
 * unpinned".  One convention inside a pinned function has no outside fact to
 * pin it: the order of the FWHT's stages (h = 1, 2, ..., 64).  Other orders
 * give the same transform up to rounding, so the tests pin the transform
 * (Sylvester H, per-stage error bound) and the order is a stated reading.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TILE 128          /* coordinates per tile [RHT] */
#define GROUP_TILES 32    /* tiles per indexed group (format reading) */
#define RANGE_LIMIT 1048576.0f      /* |y| above 2^20 is a range error */
#define SYMBOL_LIMIT (1u << 22)     /* no valid symbol reaches 2^22 */

enum { ORA_Z = 1, ORA_A2 = 2, ORA_D4 = 4, ORA_E8 = 8 };
enum {
  ORA_OK = 0, ORA_ERR_INVALID = 1, ORA_ERR_CAPACITY = 4, ORA_ERR_CORRUPT = 8,
  ORA_ERR_RANGE = 32
};

/* The oracle's own parameter block (same meaning as the library's, written
 * independently). */
typedef struct {
  int32_t lattice;            /* 1 = Z, 4 = D4, 8 = E8 */
  int32_t rice_k;             /* Rice parameter, 0..15 */
  float alpha;                /* lattice units per unit of orthonormal RHT output */
  int32_t dither;             /* 0 = off, 1 = subtractive dither */
  uint64_t dither_seed;
  uint64_t tile_base;         /* global index of the first tile of the call */
  const uint32_t *signs;      /* [n_segments][4] sign masks, bit set = -1 */
  int64_t tiles_per_segment;  /* tile t uses mask t / tiles_per_segment */
  const float *rot;           /* NULL, or [n_segments][128][128] row-major R */
} ora_params;

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al. 2011).                                       */
/* ------------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* [RHT] "D is a random sign diagonal", drawn from a seed.  Reading: one mask
 * of 128 bits per (seed, segment), from one Philox call with counter
 * (segment lo, segment hi, 0, 'SIGN'); coordinate i is negated when bit
 * (i mod 32) of word i/32 is set.  [BIAS] the cheap per-layer +-1 rotation is
 * a second diagonal applied before H; two diagonals compose by XOR of masks,
 * which the caller does. */
void oracle_make_signs(uint64_t seed, uint64_t segment, uint32_t out[4]) {
  uint32_t ctr[4] = {(uint32_t)segment, (uint32_t)(segment >> 32), 0u,
                     0x5349474Eu};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  oracle_philox4x32_10(ctr, key, out);
}

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard transform [RHT].                                          */
/* ------------------------------------------------------------------------ */
/* Unnormalised H_128 in natural (Sylvester) order, applied in place as seven
 * radix-2 stages h = 1, 2, 4, ..., 64; each output is one rounded fp32 sum or
 * difference.  The fixed stage order is part of the definition (the result is
 * bit-exact only for this order). */
void oracle_fwht128(float *x) {
  for (int h = 1; h < TILE; h <<= 1) {
    for (int i = 0; i < TILE; ++i) {
      if (i & h) continue;
      float a = x[i], b = x[i + h];
      x[i] = a + b;
      x[i + h] = a - b;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Nearest lattice points [LAT].                                            */
/* ------------------------------------------------------------------------ */
static int is_negative(float f) { return signbit(f) ? 1 : 0; }

/* Z: nearest integer, ties to even. */
int32_t oracle_nearest_z(float y) { return (int32_t)rintf(y); }

/* D4 = {v in Z^4 : sum v even} (Conway & Sloane's D_n rule): round every
 * coordinate; if the sum is odd, move the coordinate with the largest rounding
 * error (smallest index among equals) to its other neighbour, the one on the
 * side of y (an error of -0 or below counts as negative). */
void oracle_nearest_d4(const float *y, int32_t *v) {
  float err[4];
  int32_t sum = 0;
  for (int i = 0; i < 4; ++i) {
    float f = rintf(y[i]);
    v[i] = (int32_t)f;
    err[i] = y[i] - f;
    sum += v[i];
  }
  if (sum & 1) {
    int j = 0;
    for (int i = 1; i < 4; ++i)
      if (fabsf(err[i]) > fabsf(err[j])) j = i;
    v[j] += is_negative(err[j]) ? -1 : 1;
  }
}

/* [LAT] E8 with the integer embedding Lambda = 2 E8 = 2 D8 u (2 D8 + 1):
 * all coordinates of one parity and sum = 0 mod 4 (reading of "E8_int in
 * Z^8").  Closed-form decoder: the nearest point of each coset, then the
 * nearer of the two.
 *
 * Even coset 2 D8: F_i = 2 rint(y_i / 2), e_i = y_i - F_i in [-1, 1]; if
 * sum(F_i / 2) is odd, coordinate jA (largest |e|, smallest index among
 * equals) moves to the other even neighbour on the side of y.
 * Odd coset 2 D8 + 1: O_i = F_i + s_i with s_i = -1 if e_i is negative (or
 * -0), else +1; its error is 1 - |e_i|.  If sum((O_i - 1) / 2) is odd,
 * coordinate jB (smallest |e|, smallest index among equals) moves to the other
 * odd neighbour, F_jB - s_jB.
 *
 * Choosing between them.  With S = sum |e_i|, the exact difference of squared
 * distances is  dist^2(odd) - dist^2(even)
 *      = (8 - 4 pA) - 2 S + 4 pB min|e| + 4 pA max|e|
 * (pA, pB = the two parity flags), because (1 - a)^2 - a^2 = 1 - 2a, a flip
 * in the even coset costs 4 - 4a and one in the odd coset costs 4a.
 * Reading (the summary gives no formula): this difference is evaluated in
 * fp32 in exactly this order -- S summed left to right, then three fmaf
 * steps -- and the odd coset is taken only when it is negative, so exact ties
 * go to the even coset.  Rounding in S can only flip the choice when the two
 * cosets are within a few ulps of equally near. */
void oracle_nearest_e8(const float *y, int32_t *v) {
  float F[8], e[8], a[8];
  int neg[8];
  uint32_t sum_half = 0, sum_neg = 0;
  for (int i = 0; i < 8; ++i) {
    F[i] = 2.0f * rintf(0.5f * y[i]);
    e[i] = y[i] - F[i];
    a[i] = fabsf(e[i]);
    neg[i] = is_negative(e[i]);
    sum_half += (uint32_t)(int32_t)(F[i] * 0.5f);
    sum_neg += (uint32_t)neg[i];
  }
  int pA = (int)(sum_half & 1u);
  int pB = (int)((sum_half - sum_neg) & 1u);
  float S = a[0];
  for (int i = 1; i < 8; ++i) S = S + a[i];
  int jA = 0, jB = 0;
  for (int i = 1; i < 8; ++i) {
    if (a[i] > a[jA]) jA = i;
    if (a[i] < a[jB]) jB = i;
  }
  float D = fmaf(-2.0f, S, pA ? 4.0f : 8.0f);
  if (pB) D = fmaf(4.0f, a[jB], D);
  if (pA) D = fmaf(4.0f, a[jA], D);
  if (D < 0.0f) {
    for (int i = 0; i < 8; ++i) v[i] = (int32_t)F[i] + (neg[i] ? -1 : 1);
    if (pB) v[jB] = (int32_t)F[jB] - (neg[jB] ? -1 : 1);
  } else {
    for (int i = 0; i < 8; ++i) v[i] = (int32_t)F[i];
    if (pA) v[jA] += neg[jA] ? -2 : 2;
  }
}

/* [LAT] A2, the hexagonal lattice of minimal distance 1, with the integer
 * embedding (m, n) in Z^2, m = n (mod 2), for the point (m / 2, (sqrt 3 / 2) n)
 * (reading of "integer embedding" for A2: twice the first coordinate and the
 * second in units of sqrt(3)/2).  A2 is the union of two cosets of the
 * rectangular lattice Z x sqrt(3) Z, whose nearest points are found by
 * rounding each coordinate on its own:
 *   m, n even:  m = 2 rint(x),        n = 2 rint(y c)
 *   m, n odd:   m = 2 rint(x - 1/2) + 1,  n = 2 rint(y c - 1/2) + 1
 * with c = fl32(1/sqrt 3).  The nearer one wins; the squared distance of a
 * candidate is fmaf(dx, dx, fl(dy dy)) with dx = x - fl(m / 2) and
 * dy = y - fl(h n), h = fl32(sqrt(3) / 2), and exact ties go to the even coset.
 * Reading: these fp32 constants and this order are part of the definition
 * (the summary gives none). */
static const float A2_C = 0.57735026918962576f;   /* fl32(1/sqrt 3) */
static const float A2_H = 0.86602540378443865f;   /* fl32(sqrt(3)/2) */

float oracle_a2_point_y(int32_t n) { return A2_H * (float)n; }

void oracle_nearest_a2(const float *y, int32_t *v) {
  int32_t me = 2 * (int32_t)rintf(y[0]);
  int32_t ne = 2 * (int32_t)rintf(y[1] * A2_C);
  int32_t mo = 2 * (int32_t)rintf(y[0] - 0.5f) + 1;
  int32_t no = 2 * (int32_t)rintf(y[1] * A2_C - 0.5f) + 1;
  float dxe = y[0] - 0.5f * (float)me, dye = y[1] - oracle_a2_point_y(ne);
  float dxo = y[0] - 0.5f * (float)mo, dyo = y[1] - oracle_a2_point_y(no);
  float de = fmaf(dxe, dxe, dye * dye);
  float d_o = fmaf(dxo, dxo, dyo * dyo);
  if (d_o < de) { v[0] = mo; v[1] = no; }
  else { v[0] = me; v[1] = ne; }
}

/* Lattice point of a code vector: the identity for Z, D4 and 2E8; for A2 each
 * pair (m, n) is the point (m / 2, fl(h n)). */
void oracle_point(int lattice, const int32_t *v, float *pt, int n) {
  for (int i = 0; i < n; ++i) {
    if (lattice == ORA_A2) pt[i] = (i & 1) ? oracle_a2_point_y(v[i]) : 0.5f * (float)v[i];
    else pt[i] = (float)v[i];
  }
}

/* ------------------------------------------------------------------------ */
/* Subtractive dither [BIAS].                                               */
/* ------------------------------------------------------------------------ */
/* U ~ Uniform(V(Lambda)), fresh per vector, regenerated by the decoder from
 * the seed.  Reading: one Philox4x32-10 call per 8 coordinates, key = seed,
 * counter = (t lo, t hi, j, 'DITH') with t = tile_base + tile index in the
 * call and j = 0..15 the 8-coordinate group; coordinate 8j + i takes the
 * 16-bit value b_i (b_{2m} = low half of word m, b_{2m+1} = high half).
 * A point u0 uniform on a box that tiles space by the lattice (a union of
 * fundamental regions) is drawn on a grid of midpoints, then reduced:
 * u = u0 - Q(u0), which is uniform on the Voronoi cell.
 *   E8 (2E8 units): u0_i = -1 + (b + 1/2) 2^-15 for i < 7,
 *                   u0_7 = -2 + (b + 1/2) 2^-14  (box = fundamental region of 2D8,
 *                   i.e. two of 2E8).
 *   D4: u0_i = -1/2 + (b + 1/2) 2^-16 for i < 3, u0_3 = -1 + (b + 1/2) 2^-15
 *       (a fundamental region of D4).
 *   Z : u_i = -1/2 + (b + 1/2) 2^-16, already inside V(Z).
 *   A2: per pair, u0_x = -1/2 + (b + 1/2) 2^-16 and
 *       u0_y = fl(h (-1 + (b' + 1/2) 2^-15)), a point of the box
 *       [-1/2, 1/2) x [-h, h) (a fundamental region of Z x sqrt(3) Z, i.e. two
 *       cells of A2, up to the rounding of h); u = fl(u0 - point(Q(u0))).
 * All of these values except the A2 ones, and u0 - Q(u0), are exact in fp32. */
void oracle_dither(int lattice, uint64_t seed, uint64_t tile, float *u) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  for (uint32_t j = 0; j < 16; ++j) {
    uint32_t ctr[4] = {(uint32_t)tile, (uint32_t)(tile >> 32), j, 0x44495448u};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    float b[8];
    for (int m = 0; m < 4; ++m) {
      b[2 * m] = (float)(w[m] & 0xFFFFu) + 0.5f;
      b[2 * m + 1] = (float)(w[m] >> 16) + 0.5f;
    }
    float *uj = u + 8 * j;
    if (lattice == ORA_E8) {
      float u0[8];
      int32_t lam[8];
      for (int i = 0; i < 7; ++i) u0[i] = -1.0f + b[i] * 0x1p-15f;
      u0[7] = -2.0f + b[7] * 0x1p-14f;
      oracle_nearest_e8(u0, lam);
      for (int i = 0; i < 8; ++i) uj[i] = u0[i] - (float)lam[i];
    } else if (lattice == ORA_D4) {
      for (int h = 0; h < 2; ++h) {
        float u0[4];
        int32_t lam[4];
        for (int i = 0; i < 3; ++i) u0[i] = -0.5f + b[4 * h + i] * 0x1p-16f;
        u0[3] = -1.0f + b[4 * h + 3] * 0x1p-15f;
        oracle_nearest_d4(u0, lam);
        for (int i = 0; i < 4; ++i) uj[4 * h + i] = u0[i] - (float)lam[i];
      }
    } else if (lattice == ORA_A2) {
      for (int h = 0; h < 4; ++h) {
        float u0[2], pt[2];
        int32_t lam[2];
        u0[0] = -0.5f + b[2 * h] * 0x1p-16f;
        u0[1] = A2_H * (-1.0f + b[2 * h + 1] * 0x1p-15f);
        oracle_nearest_a2(u0, lam);
        oracle_point(ORA_A2, lam, pt, 2);
        uj[2 * h] = u0[0] - pt[0];
        uj[2 * h + 1] = u0[1] - pt[1];
      }
    } else {
      for (int i = 0; i < 8; ++i) uj[i] = -0.5f + b[i] * 0x1p-16f;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Fold / strip [STRIP].                                                    */
/* ------------------------------------------------------------------------ */
static uint32_t zigzag(int32_t n) {
  return n >= 0 ? 2u * (uint32_t)n : 2u * (uint32_t)(-(int64_t)n) - 1u;
}
static int32_t unzigzag(uint32_t m) {
  return (m & 1u) ? -(int32_t)(m >> 1) - 1 : (int32_t)(m >> 1);
}

/* Reading of "bits fixed by membership are stripped": every lattice vector is
 * mapped to non-negative symbols of magnitude about 2|v| (zigzag keeps the
 * sign in the low bit), arranged so that each membership-fixed bit is an
 * identifiable bit of some symbol.
 *   E8: p = v_0 mod 2 (the coset), w_i = (v_i - p)/2 (a D8 point),
 *       r = (w_0 + ... + w_6) mod 2 (= w_7 mod 2), t = (w_7 - r)/2;
 *       s_i = 2 Z(w_i) + p (i < 7), s_7 = 4 Z(t) + 2 r + p.
 *       Fixed bits: bit 0 of s_1..s_7 (= p, a copy of bit 0 of s_0) and
 *       bit 1 of s_7 (= r): 8 bits per vector = log2 [Z^8 : 2E8].
 *   D4: r = (v_0 + v_1 + v_2) mod 2, t = (v_3 - r)/2; s_i = Z(v_i) (i < 3),
 *       s_3 = 2 Z(t) + r.  Fixed bit: bit 0 of s_3.
 *   A2: per pair (m, n): p = n mod 2 (= m mod 2), w = (m - p)/2;
 *       s_0 = Z(n), s_1 = 2 Z(w) + p.  Fixed bit: bit 0 of s_1.
 *   Z : s = Z(v).  Nothing fixed. */
void oracle_fold(int lattice, const int32_t *v, uint32_t *s, int n) {
  if (lattice == ORA_E8) {
    for (int b = 0; b < n; b += 8) {
      int32_t p = v[b] & 1;
      int32_t w[8], r = 0;
      for (int i = 0; i < 8; ++i) w[i] = (v[b + i] - p) / 2;
      for (int i = 0; i < 7; ++i) r += w[i];
      r &= 1;
      int32_t t = (w[7] - r) / 2;
      for (int i = 0; i < 7; ++i) s[b + i] = 2u * zigzag(w[i]) + (uint32_t)p;
      s[b + 7] = 4u * zigzag(t) + 2u * (uint32_t)r + (uint32_t)p;
    }
  } else if (lattice == ORA_D4) {
    for (int b = 0; b < n; b += 4) {
      int32_t r = (v[b] + v[b + 1] + v[b + 2]) & 1;
      int32_t t = (v[b + 3] - r) / 2;
      for (int i = 0; i < 3; ++i) s[b + i] = zigzag(v[b + i]);
      s[b + 3] = 2u * zigzag(t) + (uint32_t)r;
    }
  } else if (lattice == ORA_A2) {
    for (int b = 0; b < n; b += 2) {
      int32_t p = v[b + 1] & 1;
      int32_t w = (v[b] - p) / 2;
      s[b] = zigzag(v[b + 1]);
      s[b + 1] = 2u * zigzag(w) + (uint32_t)p;
    }
  } else {
    for (int i = 0; i < n; ++i) s[i] = zigzag(v[i]);
  }
}

/* 1 if remainder bit `bit` of a symbol in coordinate `coord` of its vector is
 * fixed by membership and therefore not written. */
int oracle_bit_stripped(int lattice, int coord, int bit, int k) {
  if (bit >= k) return 0;
  if (lattice == ORA_E8) {
    if (bit == 0 && coord >= 1) return 1;
    if (bit == 1 && coord == 7) return 1;
  } else if (lattice == ORA_D4) {
    if (bit == 0 && coord == 3) return 1;
  } else if (lattice == ORA_A2) {
    if (bit == 0 && coord == 1) return 1;
  }
  return 0;
}

static int lattice_dim(int lattice) {
  return lattice == ORA_E8 ? 8 : (lattice == ORA_D4 ? 4 : (lattice == ORA_A2 ? 2 : 1));
}

/* Inverse of oracle_fold.  Stripped bits arrive as 0 and are restored from
 * the membership rules; bits that were not stripped (small k) must agree with
 * those rules, otherwise the vector is corrupt.  Returns 0 or ORA_ERR_CORRUPT. */
int oracle_unfold(int lattice, int k, const uint32_t *s_in, int32_t *v, int n) {
  int bad = 0;
  if (lattice == ORA_E8) {
    for (int b = 0; b < n; b += 8) {
      uint32_t s[8];
      memcpy(s, s_in + b, sizeof s);
      uint32_t p = s[0] & 1u;
      for (int i = 1; i < 8; ++i) {
        if (oracle_bit_stripped(ORA_E8, i, 0, k)) s[i] |= p;
        else if ((s[i] & 1u) != p) bad = 1;
      }
      int32_t w[8], r = 0;
      for (int i = 0; i < 7; ++i) { w[i] = unzigzag(s[i] >> 1); r += w[i]; }
      r &= 1;
      if (oracle_bit_stripped(ORA_E8, 7, 1, k)) s[7] |= (uint32_t)r << 1;
      else if (((s[7] >> 1) & 1u) != (uint32_t)r) bad = 1;
      w[7] = 2 * unzigzag(s[7] >> 2) + r;
      for (int i = 0; i < 8; ++i) v[b + i] = 2 * w[i] + (int32_t)p;
    }
  } else if (lattice == ORA_D4) {
    for (int b = 0; b < n; b += 4) {
      uint32_t s3 = s_in[b + 3];
      int32_t r = 0;
      for (int i = 0; i < 3; ++i) { v[b + i] = unzigzag(s_in[b + i]); r += v[b + i]; }
      r &= 1;
      if (oracle_bit_stripped(ORA_D4, 3, 0, k)) s3 |= (uint32_t)r;
      else if ((s3 & 1u) != (uint32_t)r) bad = 1;
      v[b + 3] = 2 * unzigzag(s3 >> 1) + r;
    }
  } else if (lattice == ORA_A2) {
    for (int b = 0; b < n; b += 2) {
      uint32_t s1 = s_in[b + 1];
      int32_t nn = unzigzag(s_in[b]);
      uint32_t p = (uint32_t)nn & 1u;
      if (oracle_bit_stripped(ORA_A2, 1, 0, k)) s1 |= p;
      else if ((s1 & 1u) != p) bad = 1;
      v[b] = 2 * unzigzag(s1 >> 1) + (int32_t)p;
      v[b + 1] = nn;
    }
  } else {
    for (int i = 0; i < n; ++i) v[i] = unzigzag(s_in[i]);
  }
  return bad ? ORA_ERR_CORRUPT : 0;
}

/* Number of remainder bits a tile writes: 128 k minus the stripped ones. */
int64_t oracle_tile_rbits(int lattice, int k) {
  int dim = lattice_dim(lattice);
  int64_t bits = 0;
  for (int j = 0; j < TILE; ++j)
    for (int b = 0; b < k; ++b)
      if (!oracle_bit_stripped(lattice, j % dim, b, k)) ++bits;
  return bits;
}

/* ------------------------------------------------------------------------ */
/* Per-tile encode and decode.                                              */
/* ------------------------------------------------------------------------ */
static const uint32_t *tile_mask(const ora_params *P, int64_t t) {
  int64_t seg = P->tiles_per_segment > 0 ? t / P->tiles_per_segment : 0;
  return P->signs + 4 * seg;
}
static int mask_bit(const uint32_t *m, int i) { return (int)((m[i >> 5] >> (i & 31)) & 1u); }

/* [BIAS] The per-layer rotation may be a full Haar-uniform (QJL) orthogonal
 * matrix instead of the cheap +-1 diagonal.  Reading: R (one per segment,
 * row-major fp32) is applied to the tile before the sign diagonal and the
 * Hadamard transform, RHT(R x); every output is one fused multiply-add chain
 * over the inputs in index order, starting from +0:
 *   z_i = fmaf(R[i][127], x[127], ... fmaf(R[i][1], x[1], fmaf(R[i][0], x[0], 0)))
 * and the decoder applies the transpose the same way (over i for each j),
 * after the inverse Hadamard transform and the sign diagonal. */
static const float *tile_rot(const ora_params *P, int64_t t) {
  int64_t seg = P->tiles_per_segment > 0 ? t / P->tiles_per_segment : 0;
  return P->rot + seg * TILE * TILE;
}
void oracle_rotate(const float *R, const float *x, float *out) {
  float z[TILE];
  for (int i = 0; i < TILE; ++i) {
    float acc = 0.0f;
    for (int j = 0; j < TILE; ++j) acc = fmaf(R[i * TILE + j], x[j], acc);
    z[i] = acc;
  }
  memcpy(out, z, sizeof z);
}
void oracle_rotate_t(const float *R, const float *y, float *out) {
  float z[TILE];
  for (int j = 0; j < TILE; ++j) {
    float acc = 0.0f;
    for (int i = 0; i < TILE; ++i) acc = fmaf(R[i * TILE + j], y[i], acc);
    z[j] = acc;
  }
  memcpy(out, z, sizeof z);
}

static float bf16_to_float(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}
static uint16_t float_to_bf16(float f) {  /* round to nearest even; finite inputs */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  uint32_t lsb = (bits >> 16) & 1u;
  return (uint16_t)((bits + 0x7FFFu + lsb) >> 16);
}

/* Scale from RHT output to lattice units.  Reading: the RHT is normalised by
 * 1/sqrt(128) so that it is orthonormal ([RHT]: "orthogonal, preserves l2"),
 * and alpha is in lattice units per unit of that output; the product is
 * formed in double and rounded once to fp32. */
float oracle_encode_scale(float alpha) { return (float)((double)alpha / sqrt(128.0)); }
float oracle_decode_scale(float alpha) { return (float)(1.0 / ((double)alpha * sqrt(128.0))); }

/* Codes of one tile.  x: 128 bf16; t: index of the tile in the call.
 * y_i = fmaf(z_i, s_enc, u_i): scale and dither in one rounding (reading:
 * the summary fixes neither; u = +0 without dither).  Range rule (reading of
 * "alpha is chosen so that codes fit"): if any y_i is NaN or |y_i| > 2^20 the
 * tile is coded as if x were 0 and ORA_ERR_RANGE is reported. */
/* z = H D (R) x and the dither u of one tile (u = +0 without dither). */
static void tile_zu(const ora_params *P, const uint16_t *x, int64_t t, float *z, float *u) {
  const uint32_t *m = tile_mask(P, t);
  float xf[TILE];
  for (int i = 0; i < TILE; ++i) xf[i] = bf16_to_float(x[i]);
  if (P->rot) oracle_rotate(tile_rot(P, t), xf, xf);
  for (int i = 0; i < TILE; ++i) z[i] = mask_bit(m, i) ? -xf[i] : xf[i];
  oracle_fwht128(z);
  if (P->dither) oracle_dither(P->lattice, P->dither_seed, P->tile_base + (uint64_t)t, u);
  else for (int i = 0; i < TILE; ++i) u[i] = 0.0f;
}

/* The lattice-domain values y of one tile (before the nearest point), with
 * the range rule applied; returns the range flag. */
static int tile_y(const ora_params *P, const uint16_t *x, int64_t t, float *y) {
  float z[TILE], u[TILE];
  tile_zu(P, x, t, z, u);
  float s = oracle_encode_scale(P->alpha);
  int flag = 0;
  for (int i = 0; i < TILE; ++i) {
    y[i] = fmaf(z[i], s, u[i]);
    if (!(fabsf(y[i]) <= RANGE_LIMIT)) flag = ORA_ERR_RANGE;
  }
  if (flag)
    for (int i = 0; i < TILE; ++i) y[i] = fmaf(0.0f, s, u[i]);
  return flag;
}

int oracle_tile_codes(const ora_params *P, const uint16_t *x, int64_t t,
                      int32_t *v) {
  float y[TILE];
  const int flag = tile_y(P, x, t, y);
  if (P->lattice == ORA_E8) {
    for (int b = 0; b < TILE; b += 8) oracle_nearest_e8(y + b, v + b);
  } else if (P->lattice == ORA_D4) {
    for (int b = 0; b < TILE; b += 4) oracle_nearest_d4(y + b, v + b);
  } else if (P->lattice == ORA_A2) {
    for (int b = 0; b < TILE; b += 2) oracle_nearest_a2(y + b, v + b);
  } else {
    for (int i = 0; i < TILE; ++i) v[i] = oracle_nearest_z(y[i]);
  }
  return flag;
}

/* Reconstruction of one tile from its codes: e_i = v_i - u_i, the same FWHT,
 * x_i = fl(z_i * s_dec), then the sign mask (H is symmetric and H H = 128 I,
 * so this inverts the forward transform up to rounding). */
void oracle_tile_reconstruct(const ora_params *P, const int32_t *v, int64_t t,
                             float *out) {
  const uint32_t *m = tile_mask(P, t);
  float u[TILE], z[TILE];
  if (P->dither) oracle_dither(P->lattice, P->dither_seed, P->tile_base + (uint64_t)t, u);
  else for (int i = 0; i < TILE; ++i) u[i] = 0.0f;
  float pt[TILE];
  oracle_point(P->lattice, v, pt, TILE);
  for (int i = 0; i < TILE; ++i) z[i] = pt[i] - u[i];
  oracle_fwht128(z);
  float s = oracle_decode_scale(P->alpha);
  for (int i = 0; i < TILE; ++i) {
    float r = z[i] * s;
    out[i] = mask_bit(m, i) ? -r : r;
  }
  if (P->rot) oracle_rotate_t(tile_rot(P, t), out, out);
}

/* ------------------------------------------------------------------------ */
/* Stream format (reading; the summary gives none).                         */
/* ------------------------------------------------------------------------ */
/* Tiles are indexed in groups of 32 consecutive tiles; every group starts on a
 * 32-bit word boundary.  A group holds, in order:
 *   R-area: for each tile of the group, the kept remainder bits of its 128
 *           symbols (symbol order = coordinate order; bits from k-1 down to 0,
 *           stripped bits skipped);
 *   U-area: for each tile, for each symbol, q = s >> k zeros then a one;
 *   zero padding up to the next word.
 * This is the same set of Rice codewords as a plain concatenation, reordered
 * so that remainders sit at fixed positions and unary terminators can be
 * counted in parallel.  Bit b of a group is bit 31 - (b mod 32) of word b/32.
 * offsets[g] = word index of group g; offsets[n_groups] = total words. */

static void put_bit(uint32_t *words, uint64_t cap, uint64_t base, uint64_t b, int bit) {
  uint64_t w = base + (b >> 5);
  if (bit && w < cap) words[w] |= 0x80000000u >> (b & 31);
}

typedef void (*range_fn)(void *ctx, int64_t begin, int64_t end);
typedef struct { range_fn fn; void *ctx; int64_t begin, end; } job_t;
static void *run_job(void *arg) { job_t *j = (job_t *)arg; j->fn(j->ctx, j->begin, j->end); return NULL; }

/* Plain parallel-for over [0, n): contiguous chunks, one per thread. */
static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads == 1 || n < 2) { fn(ctx, 0, n); return; }
  pthread_t th[256];
  job_t jobs[256];
  int64_t chunk = (n + nthreads - 1) / nthreads;
  int used = 0;
  for (int i = 0; i < nthreads; ++i) {
    int64_t b = i * chunk, e = b + chunk < n ? b + chunk : n;
    if (b >= e) break;
    jobs[i].fn = fn; jobs[i].ctx = ctx; jobs[i].begin = b; jobs[i].end = e;
    if (pthread_create(&th[i], NULL, run_job, &jobs[i]) != 0) { fn(ctx, b, e); jobs[i].fn = NULL; }
    used = i + 1;
  }
  for (int i = 0; i < used; ++i) if (jobs[i].fn) pthread_join(th[i], NULL);
}

typedef struct {
  const ora_params *P;
  const uint16_t *x;
  int64_t n_tiles;
  uint32_t *sym;        /* [n_tiles][128] */
  uint64_t *ubits;      /* [n_tiles] unary bits per tile */
  uint32_t *flags;      /* [n_tiles] */
  int32_t *v_out;       /* [n_tiles][128] or NULL */
  uint32_t *stream;
  uint64_t cap;
  const uint64_t *offsets;
  int64_t rbits;
} enc_ctx;

static void enc_symbols(void *c, int64_t b, int64_t e) {
  enc_ctx *C = (enc_ctx *)c;
  int32_t v[TILE];
  for (int64_t t = b; t < e; ++t) {
    C->flags[t] = (uint32_t)oracle_tile_codes(C->P, C->x + t * TILE, t, v);
    if (C->v_out) memcpy(C->v_out + t * TILE, v, sizeof v);
    uint32_t *s = C->sym + t * TILE;
    oracle_fold(C->P->lattice, v, s, TILE);
    uint64_t u = 0;
    for (int j = 0; j < TILE; ++j) u += (uint64_t)(s[j] >> C->P->rice_k) + 1u;
    C->ubits[t] = u;
  }
}

static void enc_write(void *c, int64_t gb, int64_t ge) {
  enc_ctx *C = (enc_ctx *)c;
  int k = C->P->rice_k, dim = lattice_dim(C->P->lattice);
  for (int64_t g = gb; g < ge; ++g) {
    uint64_t base = C->offsets[g], words = C->offsets[g + 1] - base;
    for (uint64_t w = 0; w < words; ++w)
      if (base + w < C->cap) C->stream[base + w] = 0u;
    int64_t t0 = g * GROUP_TILES;
    int64_t t1 = t0 + GROUP_TILES < C->n_tiles ? t0 + GROUP_TILES : C->n_tiles;
    uint64_t b = 0;
    for (int64_t t = t0; t < t1; ++t) {            /* R-area */
      const uint32_t *s = C->sym + t * TILE;
      for (int j = 0; j < TILE; ++j)
        for (int bit = k - 1; bit >= 0; --bit)
          if (!oracle_bit_stripped(C->P->lattice, j % dim, bit, k))
            put_bit(C->stream, C->cap, base, b++, (int)((s[j] >> bit) & 1u));
    }
    for (int64_t t = t0; t < t1; ++t) {            /* U-area */
      const uint32_t *s = C->sym + t * TILE;
      for (int j = 0; j < TILE; ++j) {
        b += s[j] >> k;                            /* q zeros (already 0) */
        put_bit(C->stream, C->cap, base, b++, 1);
      }
    }
  }
}

static int params_ok(const ora_params *P) {
  if (!P || !P->signs) return 0;
  if (P->lattice != ORA_Z && P->lattice != ORA_A2 && P->lattice != ORA_D4 &&
      P->lattice != ORA_E8)
    return 0;
  if (P->rice_k < 0 || P->rice_k > 15) return 0;
  if (!(P->alpha > 0.0f) || !isfinite(P->alpha)) return 0;
  if (P->dither != 0 && P->dither != 1) return 0;
  if (P->tiles_per_segment <= 0) return 0;
  return 1;
}

int64_t oracle_n_groups(int64_t n_tiles) { return (n_tiles + GROUP_TILES - 1) / GROUP_TILES; }

/* Encode n_tiles tiles.  offsets needs n_groups + 1 entries.  Words at index
 * >= cap_words are not written (status gets ORA_ERR_CAPACITY), but offsets
 * are always complete.  Optionally returns per-tile codes (v_out, may be NULL)
 * and payload bits per tile (tile_bits, may be NULL).  Returns the total
 * number of words, or -1 for invalid arguments. */
int64_t oracle_encode(const ora_params *P, const uint16_t *x, int64_t n_tiles,
                      uint32_t *stream, uint64_t cap_words, uint64_t *offsets,
                      uint32_t *status, int32_t *v_out, uint64_t *tile_bits,
                      int nthreads) {
  if (!params_ok(P) || n_tiles < 0 || !offsets || !status) return -1;
  int64_t ng = oracle_n_groups(n_tiles);
  enc_ctx C;
  memset(&C, 0, sizeof C);
  C.P = P; C.x = x; C.n_tiles = n_tiles; C.stream = stream; C.cap = stream ? cap_words : 0;
  C.v_out = v_out;
  C.rbits = oracle_tile_rbits(P->lattice, P->rice_k);
  C.sym = (uint32_t *)malloc(sizeof(uint32_t) * TILE * (size_t)(n_tiles > 0 ? n_tiles : 1));
  C.ubits = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n_tiles > 0 ? n_tiles : 1));
  C.flags = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(n_tiles > 0 ? n_tiles : 1));
  if (!C.sym || !C.ubits || !C.flags) { free(C.sym); free(C.ubits); free(C.flags); return -1; }
  parallel_for(n_tiles, nthreads, enc_symbols, &C);
  uint32_t st = 0;
  offsets[0] = 0;
  for (int64_t g = 0; g < ng; ++g) {
    int64_t t0 = g * GROUP_TILES;
    int64_t t1 = t0 + GROUP_TILES < n_tiles ? t0 + GROUP_TILES : n_tiles;
    uint64_t bits = 0;
    for (int64_t t = t0; t < t1; ++t) {
      bits += (uint64_t)C.rbits + C.ubits[t];
      st |= C.flags[t];
      if (tile_bits) tile_bits[t] = (uint64_t)C.rbits + C.ubits[t];
    }
    offsets[g + 1] = offsets[g] + (bits + 31) / 32;
  }
  C.offsets = offsets;
  if (stream) parallel_for(ng, nthreads, enc_write, &C);
  if (offsets[ng] > cap_words) st |= ORA_ERR_CAPACITY;
  *status |= st;
  int64_t total = (int64_t)offsets[ng];
  free(C.sym); free(C.ubits); free(C.flags);
  return total;
}

/* Payload bits of an encode (sum of tile bits, no padding, no index); used
 * by rate calibration. */
int64_t oracle_payload_bits(const ora_params *P, const uint16_t *x, int64_t n_tiles,
                            int nthreads) {
  int64_t ng = oracle_n_groups(n_tiles);
  uint64_t *off = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(ng + 1));
  uint64_t *tb = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n_tiles > 0 ? n_tiles : 1));
  uint32_t st = 0;
  int64_t total = -1;
  if (off && tb && oracle_encode(P, x, n_tiles, NULL, 0, off, &st, NULL, tb, nthreads) >= 0) {
    total = 0;
    for (int64_t t = 0; t < n_tiles; ++t) total += (int64_t)tb[t];
  }
  free(off); free(tb);
  return total;
}

/* -------------------------------- decode -------------------------------- */
static int get_bit(const uint32_t *words, uint64_t base, uint64_t b) {
  return (int)((words[base + (b >> 5)] >> (31 - (b & 31))) & 1u);
}

typedef struct {
  const ora_params *P;
  const uint32_t *stream;
  uint64_t stream_words;
  const uint64_t *offsets;
  int64_t n_tiles;
  float *out_f32;
  uint16_t *out_bf16;
  int32_t *v_out;
  uint32_t *gflags;
} dec_ctx;

/* Parse group g into symbols; returns 0 or ORA_ERR_CORRUPT. */
static int parse_group(const dec_ctx *C, int64_t g, uint32_t *sym /*[32][128]*/) {
  const ora_params *P = C->P;
  int k = P->rice_k, dim = lattice_dim(P->lattice);
  uint64_t base = C->offsets[g];
  if (C->offsets[g + 1] < base || C->offsets[g + 1] > C->stream_words) return ORA_ERR_CORRUPT;
  uint64_t nbits = (C->offsets[g + 1] - base) * 32u;
  int64_t t0 = g * GROUP_TILES;
  int64_t t1 = t0 + GROUP_TILES < C->n_tiles ? t0 + GROUP_TILES : C->n_tiles;
  int nt = (int)(t1 - t0);
  uint64_t b = 0;
  for (int t = 0; t < nt; ++t)
    for (int j = 0; j < TILE; ++j) {
      uint32_t s = 0;
      for (int bit = k - 1; bit >= 0; --bit) {
        if (oracle_bit_stripped(P->lattice, j % dim, bit, k)) continue;
        if (b >= nbits) return ORA_ERR_CORRUPT;
        s |= (uint32_t)get_bit(C->stream, base, b++) << bit;
      }
      sym[t * TILE + j] = s;
    }
  uint32_t qmax = (SYMBOL_LIMIT - 1u) >> k;
  for (int t = 0; t < nt; ++t)
    for (int j = 0; j < TILE; ++j) {
      uint32_t q = 0;
      for (;;) {
        if (b >= nbits) return ORA_ERR_CORRUPT;
        if (get_bit(C->stream, base, b++)) break;
        if (++q > qmax) return ORA_ERR_CORRUPT;
      }
      sym[t * TILE + j] |= q << k;
    }
  if ((b + 31) / 32 != nbits / 32) return ORA_ERR_CORRUPT;   /* exact length */
  for (; b < nbits; ++b)
    if (get_bit(C->stream, base, b)) return ORA_ERR_CORRUPT;  /* zero padding */
  return 0;
}

static void dec_groups(void *c, int64_t gb, int64_t ge) {
  dec_ctx *C = (dec_ctx *)c;
  uint32_t *sym = (uint32_t *)malloc(sizeof(uint32_t) * TILE * GROUP_TILES);
  int32_t v[TILE];
  float x[TILE];
  for (int64_t g = gb; g < ge; ++g) {
    int64_t t0 = g * GROUP_TILES;
    int64_t t1 = t0 + GROUP_TILES < C->n_tiles ? t0 + GROUP_TILES : C->n_tiles;
    int bad = sym ? parse_group(C, g, sym) : ORA_ERR_CORRUPT;
    for (int64_t t = t0; t < t1 && !bad; ++t)
      bad |= oracle_unfold(C->P->lattice, C->P->rice_k, sym + (t - t0) * TILE, v, TILE);
    for (int64_t t = t0; t < t1; ++t) {
      if (bad) {
        memset(v, 0, sizeof v);
        for (int i = 0; i < TILE; ++i) x[i] = 0.0f;
      } else {
        oracle_unfold(C->P->lattice, C->P->rice_k, sym + (t - t0) * TILE, v, TILE);
        oracle_tile_reconstruct(C->P, v, t, x);
      }
      if (C->v_out) memcpy(C->v_out + t * TILE, v, sizeof v);
      if (C->out_f32) memcpy(C->out_f32 + t * TILE, x, sizeof x);
      if (C->out_bf16)
        for (int i = 0; i < TILE; ++i) C->out_bf16[t * TILE + i] = float_to_bf16(x[i]);
    }
    C->gflags[g] = (uint32_t)bad;
  }
  free(sym);
}

/* Decode n_tiles tiles from stream[0 .. stream_words).  Either output may be
 * NULL.  A group that fails any check (including index entries outside the
 * stream) decodes to zeros and sets ORA_ERR_CORRUPT.  Returns 0, or -1 for
 * invalid arguments. */
int oracle_decode(const ora_params *P, const uint32_t *stream, uint64_t stream_words,
                  const uint64_t *offsets,
                  int64_t n_tiles, float *out_f32, uint16_t *out_bf16, int32_t *v_out,
                  uint32_t *status, int nthreads) {
  if (!params_ok(P) || n_tiles < 0 || !offsets || !status || (!stream && n_tiles > 0)) return -1;
  int64_t ng = oracle_n_groups(n_tiles);
  dec_ctx C;
  C.P = P; C.stream = stream; C.stream_words = stream_words; C.offsets = offsets;
  C.n_tiles = n_tiles;
  C.out_f32 = out_f32; C.out_bf16 = out_bf16; C.v_out = v_out;
  C.gflags = (uint32_t *)calloc((size_t)(ng > 0 ? ng : 1), sizeof(uint32_t));
  if (!C.gflags) return -1;
  parallel_for(ng, nthreads, dec_groups, &C);
  uint32_t st = 0;
  for (int64_t g = 0; g < ng; ++g) st |= C.gflags[g];
  free(C.gflags);
  *status |= st;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention scores from compressed K [FUSED].                              */
/* ------------------------------------------------------------------------ */
/* K tile for (kv head h, token t) is tile h * n_tokens + t.  Query head hq
 * reads kv head hq / (Hq / n_kv_heads).  scores[b][hq][t] =
 * sum_d q[b][hq][d] * Khat[h][t][d], with Khat the fp32 decode above; the sum
 * is taken in double and stored as fp32.  Khat: [n_kv_heads * n_tokens][128]. */
typedef struct {
  const float *khat;
  const uint16_t *q;
  int n_kv, B, Hq;
  int64_t T;
  float *scores;
} sc_ctx;

static void scores_rows(void *c, int64_t rb, int64_t re) {
  sc_ctx *C = (sc_ctx *)c;
  int group = C->Hq / C->n_kv;
  for (int64_t row = rb; row < re; ++row) {       /* row = b * Hq + hq */
    int hq = (int)(row % C->Hq);
    int h = hq / group;
    const uint16_t *qv = C->q + row * TILE;
    double qd[TILE];
    for (int d = 0; d < TILE; ++d) qd[d] = (double)bf16_to_float(qv[d]);
    for (int64_t t = 0; t < C->T; ++t) {
      const float *kv = C->khat + ((int64_t)h * C->T + t) * TILE;
      double acc = 0.0;
      for (int d = 0; d < TILE; ++d) acc += qd[d] * (double)kv[d];
      C->scores[row * C->T + t] = (float)acc;
    }
  }
}

int oracle_scores(const float *khat, int n_kv_heads, int64_t n_tokens, const uint16_t *q,
                  int B, int Hq, float *scores, int nthreads) {
  if (n_kv_heads <= 0 || Hq <= 0 || B < 0 || Hq % n_kv_heads != 0 || n_tokens < 0) return -1;
  sc_ctx C = {khat, q, n_kv_heads, B, Hq, n_tokens, scores};
  parallel_for((int64_t)B * Hq, nthreads, scores_rows, &C);
  return 0;
}

/* Exposed limits so that tests can read the format constants. */
/* ------------------------------------------------------------------------ */
/* Diagnostic, no counterpart in the method: how often the E8 coset choice   */
/* by the fp32 linear identity (oracle_nearest_e8) differs from the plain    */
/* rule -- both cosets' nearest points by Conway & Sloane's D_n decoder on   */
/* a = y/2 and a - 1/2, then the two fp32 squared distances summed left to   */
/* right, the odd coset only when strictly nearer.                            */
/* ------------------------------------------------------------------------ */
static void dn8_nearest(const float *b, float *f) {
  float best = -1.0f;
  int j = 0, par = 0;
  for (int i = 0; i < 8; ++i) {
    f[i] = rintf(b[i]);
    par ^= ((int64_t)f[i]) & 1;
    const float d = fabsf(b[i] - f[i]);
    if (d > best) { best = d; j = i; }
  }
  if (par) f[j] += (b[j] >= f[j]) ? 1.0f : -1.0f;
}

void oracle_e8_plain(const float *y, int32_t *v) {
  float a[8], a2[8], A[8], B[8];
  for (int i = 0; i < 8; ++i) { a[i] = 0.5f * y[i]; a2[i] = a[i] - 0.5f; }
  dn8_nearest(a, A);
  dn8_nearest(a2, B);
  float dA = 0.0f, dB = 0.0f;
  for (int i = 0; i < 8; ++i) {
    A[i] = 2.0f * A[i];
    B[i] = 2.0f * B[i] + 1.0f;
    const float da = y[i] - A[i], db = y[i] - B[i];
    dA = dA + da * da;
    dB = dB + db * db;
  }
  const float *w = (dB < dA) ? B : A;
  for (int i = 0; i < 8; ++i) v[i] = (int32_t)w[i];
}

typedef struct {
  const ora_params *P;
  const uint16_t *x;
  pthread_mutex_t mu;
  int64_t vectors, differ, coset_differ;
  double dist_sum, max_abs;   /* sum of exact (double) dist^2(plain) - dist^2(oracle) */
} census_ctx;

static void census_range(void *c, int64_t b, int64_t e) {
  census_ctx *C = (census_ctx *)c;
  int64_t nv = 0, nd = 0, nc = 0;
  double ds = 0.0, mx = 0.0;
  float y[TILE];
  for (int64_t t = b; t < e; ++t) {
    tile_y(C->P, C->x + t * TILE, t, y);
    for (int q = 0; q < TILE; q += 8) {
      int32_t vo[8], vp[8];
      oracle_nearest_e8(y + q, vo);
      oracle_e8_plain(y + q, vp);
      ++nv;
      if (memcmp(vo, vp, sizeof vo) != 0) {
        ++nd;
        if (((vo[0] ^ vp[0]) & 1) != 0) ++nc;
        double d2o = 0.0, d2p = 0.0;
        for (int i = 0; i < 8; ++i) {
          const double eo = (double)y[q + i] - vo[i], ep = (double)y[q + i] - vp[i];
          d2o += eo * eo;
          d2p += ep * ep;
        }
        ds += d2p - d2o;
        if (fabs(d2p - d2o) > mx) mx = fabs(d2p - d2o);
      }
    }
  }
  pthread_mutex_lock(&C->mu);
  C->vectors += nv;
  C->differ += nd;
  C->coset_differ += nc;
  C->dist_sum += ds;
  if (mx > C->max_abs) C->max_abs = mx;
  pthread_mutex_unlock(&C->mu);
}

/* out[0] = 8-vectors coded, out[1] = vectors whose codes differ between the
 * two rules, out[2] = of those, vectors whose coset differs; dist[0] = sum
 * over the differing vectors of the exact squared distance to the plain
 * rule's point minus that to the oracle's, dist[1] = the largest |.| of one
 * vector.  E8 only. */
int oracle_e8_rule_census(const ora_params *P, const uint16_t *x, int64_t n_tiles, int64_t *out,
                          double *dist, int nthreads) {
  if (!params_ok(P) || P->lattice != ORA_E8 || n_tiles < 0) return -1;
  census_ctx C;
  memset(&C, 0, sizeof C);
  C.P = P;
  C.x = x;
  pthread_mutex_init(&C.mu, NULL);
  parallel_for(n_tiles, nthreads, census_range, &C);
  pthread_mutex_destroy(&C.mu);
  out[0] = C.vectors;
  out[1] = C.differ;
  out[2] = C.coset_differ;
  dist[0] = C.dist_sum;
  dist[1] = C.max_abs;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Diagnostic, no counterpart in the method: how often the scale and the     */
/* dither rounded once, y = fl(z s_enc + u) (the reading the codec takes),    */
/* and rounded twice, y' = fl(fl(z s_enc) + u), lead to different lattice     */
/* points, and which of the two points is nearer to the exact z s_enc + u.    */
/* ------------------------------------------------------------------------ */
/* Codes of one vector of the lattice (dim coordinates). */
static void vector_codes(int lattice, const float *y, int32_t *v) {
  if (lattice == ORA_E8) oracle_nearest_e8(y, v);
  else if (lattice == ORA_D4) oracle_nearest_d4(y, v);
  else if (lattice == ORA_A2) oracle_nearest_a2(y, v);
  else v[0] = oracle_nearest_z(y[0]);
}

/* Squared distance (double) from the exact values ye to the point coded by
 * v: the codes themselves, except A2's (m, n) = the point (m/2, h n). */
static double point_dist2(int lattice, const double *ye, const int32_t *v) {
  const int d = lattice_dim(lattice);
  double s = 0.0;
  for (int i = 0; i < d; ++i) {
    double pt = (double)v[i];
    if (lattice == ORA_A2) pt = (i == 0) ? 0.5 * v[0] : (double)oracle_a2_point_y(v[1]);
    s += (ye[i] - pt) * (ye[i] - pt);
  }
  return s;
}

typedef struct {
  const ora_params *P;
  const uint16_t *x;
  pthread_mutex_t mu;
  int64_t vectors, differ, skipped;
  double dist_sum, max_abs;
} rnd_ctx;

static void rounding_range(void *c, int64_t b, int64_t e) {
  rnd_ctx *C = (rnd_ctx *)c;
  const int lat = C->P->lattice, d = lattice_dim(lat);
  const float s = oracle_encode_scale(C->P->alpha);
  int64_t nv = 0, nd = 0, nk = 0;
  double ds = 0.0, mx = 0.0;
  float z[TILE], u[TILE], y1[TILE], y2[TILE];
  for (int64_t t = b; t < e; ++t) {
    tile_zu(C->P, C->x + t * TILE, t, z, u);
    int out = 0;
    for (int i = 0; i < TILE; ++i) {
      y1[i] = fmaf(z[i], s, u[i]);
      const float a = z[i] * s;           /* two roundings (no contraction here) */
      y2[i] = a + u[i];
      if (!(fabsf(y1[i]) <= RANGE_LIMIT) || !(fabsf(y2[i]) <= RANGE_LIMIT)) out = 1;
    }
    if (out) { ++nk; continue; }          /* the range rule decides such tiles */
    for (int q = 0; q < TILE; q += d) {
      int32_t v1[8], v2[8];
      vector_codes(lat, y1 + q, v1);
      vector_codes(lat, y2 + q, v2);
      ++nv;
      if (memcmp(v1, v2, sizeof(int32_t) * d) != 0) {
        double ye[8];
        for (int i = 0; i < d; ++i) ye[i] = (double)z[q + i] * (double)s + (double)u[q + i];
        const double diff = point_dist2(lat, ye, v2) - point_dist2(lat, ye, v1);
        ++nd;
        ds += diff;
        if (fabs(diff) > mx) mx = fabs(diff);
      }
    }
  }
  pthread_mutex_lock(&C->mu);
  C->vectors += nv;
  C->differ += nd;
  C->skipped += nk;
  C->dist_sum += ds;
  if (mx > C->max_abs) C->max_abs = mx;
  pthread_mutex_unlock(&C->mu);
}

/* out[0] = lattice vectors compared, out[1] = vectors whose points differ
 * between the two roundings, out[2] = tiles left out because either reading
 * trips the range rule; dist[0] = sum over the differing vectors of the
 * exact squared distance from z s_enc + u to the twice-rounded reading's
 * point minus that to the once-rounded reading's point (positive: the
 * codec's reading is nearer), dist[1] = the largest |.| of one vector. */
int oracle_scale_rounding_census(const ora_params *P, const uint16_t *x, int64_t n_tiles,
                                 int64_t *out, double *dist, int nthreads) {
  if (!params_ok(P) || n_tiles < 0) return -1;
  rnd_ctx C;
  memset(&C, 0, sizeof C);
  C.P = P;
  C.x = x;
  pthread_mutex_init(&C.mu, NULL);
  parallel_for(n_tiles, nthreads, rounding_range, &C);
  pthread_mutex_destroy(&C.mu);
  out[0] = C.vectors;
  out[1] = C.differ;
  out[2] = C.skipped;
  dist[0] = C.dist_sum;
  dist[1] = C.max_abs;
  return 0;
}

int oracle_group_tiles(void) { return GROUP_TILES; }
float oracle_range_limit(void) { return RANGE_LIMIT; }
uint32_t oracle_symbol_limit(void) { return SYMBOL_LIMIT; }

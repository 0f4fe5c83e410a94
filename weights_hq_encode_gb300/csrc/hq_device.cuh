// hq_device.cuh -- device primitives of the HyperQuant tile codec (sm_103a).
//
// Every floating-point step here is written with explicit round-to-nearest
// intrinsics (__fadd_rn, __fmul_rn, __fmaf_rn) and the library is built with
// --fmad=false, so each sum, product and fused multiply-add rounds exactly
// once where it is written; codes and bitstreams are therefore reproducible
// bit for bit on any IEEE fp32 implementation that follows the same steps.
#pragma once
#include <cstdint>

namespace hq {

constexpr int kTile = 128;
constexpr int kGroupTiles = 32;
constexpr float kRangeLimit = 1048576.0f;        // |y| > 2^20 -> range error
constexpr uint32_t kSymbolLimit = 1u << 22;      // no valid symbol reaches 2^22
constexpr float kMagic1 = 12582912.0f;           // 1.5 * 2^23: round to integer
constexpr float kMagic2 = 25165824.0f;           // 1.5 * 2^24: round to even integer

// ---------------------------------------------------------------- Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
// (SC'11): 10 rounds of the 4x32 bijection with multipliers D2511F53 and
// CD9E8D57 and Weyl key increments 9E3779B9 and BB67AE85.
__device__ __forceinline__ uint4 philox10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

constexpr uint32_t kDitherTag = 0x44495448u;   // 'DITH'

// 16-bit uniform b_i (i = 0..7) of one 8-coordinate group, as the float b + 1/2.
__device__ __forceinline__ void dither_halves(uint64_t seed, uint64_t tile, uint32_t j,
                                              float b[8]) {
  uint4 w = philox10(make_uint4((uint32_t)tile, (uint32_t)(tile >> 32), j, kDitherTag),
                     (uint32_t)seed, (uint32_t)(seed >> 32));
  uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    b[2 * m] = __fadd_rn((float)(ws[m] & 0xFFFFu), 0.5f);
    b[2 * m + 1] = __fadd_rn((float)(ws[m] >> 16), 0.5f);
  }
}

// ---------------------------------------------------------------- FWHT-128
// Unnormalised Walsh-Hadamard transform, natural (Sylvester) order, stages
// h = 1, 2, ..., 64 in that order (Method 1).
__device__ __forceinline__ void fwht128(float x[128]) {
#pragma unroll
  for (int h = 1; h < 128; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 128; ++i) {
      if (i & h) continue;
      float a = x[i], b = x[i + h];
      x[i] = __fadd_rn(a, b);
      x[i + h] = __fsub_rn(a, b);
    }
  }
}

// The same transform with a tile spread over 8 consecutive lanes, lane r of
// the tile holding coordinates 16r .. 16r+15: stages h = 1, 2, 4, 8 stay in
// registers, stages 16, 32, 64 pair lane r with lane r ^ 1, r ^ 2, r ^ 4.
// The lower coordinate of a pair gets fl(a + b), the upper fl(a - b), exactly
// as in the single-thread order (one rounding each, same stage order).
__device__ __forceinline__ void fwht128_x8(float x[16], int r) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      float a = x[i], b = x[i + h];
      x[i] = __fadd_rn(a, b);
      x[i + h] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    const float sg = (r & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float o = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = __fmaf_rn(x[i], sg, o);        // lower: mine + other; upper: other - mine
    }
  }
}

// 1 << n for n < 32, and 0 for n >= 32 (PTX shl clamps the shift amount).
__device__ __forceinline__ uint32_t bit_at(uint32_t n) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(1u), "r"(n));
  return r;
}

// ---------------------------------------------------------------- lattices
__device__ __forceinline__ uint32_t fbits(float f) { return __float_as_uint(f); }
__device__ __forceinline__ uint32_t zigzag(int32_t n) {
  return ((uint32_t)n << 1) ^ (uint32_t)(n >> 31);
}
__device__ __forceinline__ int32_t unzigzag(uint32_t m) {
  return (int32_t)(m >> 1) ^ -(int32_t)(m & 1u);
}

// Nearest point of 2E8 = 2D8 u (2D8 + 1) (Method 2): the even-coset point is
// built from F = 2 rint(y/2), the odd one from F + sign(e); the nearer is
// chosen by the exact identity
//   d^2(odd) - d^2(even) = (8 - 4pA) - 2 S + 4 pB min|e| + 4 pA max|e|
// evaluated in fp32 in a fixed order (S summed left to right).  The result is
// returned as the coset flag `odd` plus, per coordinate, the even-coset half
// k_i = F_i / 2, the error sign neg_i and the index of the one moved
// coordinate (jfix, or -1).
struct E8Point {
  int32_t k[8];      // F_i / 2
  uint32_t neg;      // bit i: e_i negative (sign bit set)
  int jfix;          // coordinate moved by the parity fix of the chosen coset, or -1
  bool odd;          // chosen coset is 2D8 + 1
};

__device__ __forceinline__ E8Point nearest_e8(const float y[8]) {
  E8Point r;
  float a[8];
  uint32_t par = 0, neg = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float T = __fadd_rn(y[i], kMagic2);
    float F = __fsub_rn(T, kMagic2);
    float e = __fsub_rn(y[i], F);
    a[i] = fabsf(e);
    r.k[i] = (int32_t)(fbits(T) - fbits(kMagic2));
    par ^= fbits(T);
    neg |= (fbits(e) >> 31) << i;
  }
  uint32_t pA = par & 1u;
  uint32_t pB = pA ^ (__popc(neg) & 1u);
  float S = a[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) S = __fadd_rn(S, a[i]);
  int jA = 0, jB = 0;
  float mx = a[0], mn = a[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    if (a[i] > mx) { mx = a[i]; jA = i; }
    if (a[i] < mn) { mn = a[i]; jB = i; }
  }
  float D = __fmaf_rn(-2.0f, S, pA ? 4.0f : 8.0f);
  if (pB) D = __fmaf_rn(4.0f, mn, D);
  if (pA) D = __fmaf_rn(4.0f, mx, D);
  r.odd = D < 0.0f;
  r.neg = neg;
  r.jfix = r.odd ? (pB ? jB : -1) : (pA ? jA : -1);
  return r;
}

// Lattice point (integers) of an E8Point.
__device__ __forceinline__ int32_t e8_coord(const E8Point &p, int i) {
  int32_t F = 2 * p.k[i];
  int s = ((p.neg >> i) & 1u) ? -1 : 1;
  if (p.odd) return (i == p.jfix) ? F - s : F + s;
  return (i == p.jfix) ? F + 2 * s : F;
}

// D4 = {v : sum v even} (Conway & Sloane's D_n rule).
__device__ __forceinline__ void nearest_d4(const float y[4], int32_t v[4]) {
  float a[4];
  uint32_t par = 0, neg = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float T = __fadd_rn(y[i], kMagic1);
    float f = __fsub_rn(T, kMagic1);
    float e = __fsub_rn(y[i], f);
    a[i] = fabsf(e);
    v[i] = (int32_t)(fbits(T) - fbits(kMagic1));
    par ^= fbits(T);
    neg |= (fbits(e) >> 31) << i;
  }
  if (par & 1u) {
    int j = 0;
    float mx = a[0];
#pragma unroll
    for (int i = 1; i < 4; ++i)
      if (a[i] > mx) { mx = a[i]; j = i; }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i == j) v[i] += ((neg >> i) & 1u) ? -1 : 1;
  }
}

__device__ __forceinline__ int32_t nearest_z(float y) {
  return (int32_t)(fbits(__fadd_rn(y, kMagic1)) - fbits(kMagic1));
}

// ---------------------------------------------------------------- dither
// U ~ Uniform(V(Lambda)) for the 8 coordinates of group j of a tile (Method 4):
// a grid point u0 of a box that tiles space by the lattice, minus Q(u0).
template <int LAT>
__device__ __forceinline__ void dither8(uint64_t seed, uint64_t tile, uint32_t j, float u[8]) {
  float b[8];
  dither_halves(seed, tile, j, b);
  if (LAT == 8) {
    float u0[8];
#pragma unroll
    for (int i = 0; i < 7; ++i) u0[i] = __fadd_rn(-1.0f, __fmul_rn(b[i], 0x1p-15f));
    u0[7] = __fadd_rn(-2.0f, __fmul_rn(b[7], 0x1p-14f));
    E8Point p = nearest_e8(u0);
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = __fsub_rn(u0[i], (float)e8_coord(p, i));
  } else if (LAT == 4) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float u0[4];
      int32_t lam[4];
#pragma unroll
      for (int i = 0; i < 3; ++i) u0[i] = __fadd_rn(-0.5f, __fmul_rn(b[4 * h + i], 0x1p-16f));
      u0[3] = __fadd_rn(-1.0f, __fmul_rn(b[4 * h + 3], 0x1p-15f));
      nearest_d4(u0, lam);
#pragma unroll
      for (int i = 0; i < 4; ++i) u[4 * h + i] = __fsub_rn(u0[i], (float)lam[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = __fadd_rn(-0.5f, __fmul_rn(b[i], 0x1p-16f));
  }
}

// ---------------------------------------------------------------- fold / strip
// Symbols of one 8-coordinate group (Method 3).  E8: p = coset, w = (v - p)/2,
// r = parity(w0..w6), t = (w7 - r)/2; s_i = 2Z(w_i) + p, s_7 = 4Z(t) + 2r + p.
// D4 (two vectors): r = parity(v0+v1+v2), t = (v3 - r)/2, s_3 = 2Z(t) + r.
template <int LAT>
__device__ __forceinline__ void quantize_fold8(const float y[8], uint32_t s[8]) {
  if (LAT == 8) {
    E8Point p = nearest_e8(y);
    int32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int32_t ng = (int32_t)((p.neg >> i) & 1u);
      int32_t fix = (i == p.jfix) ? 1 : 0;
      // even coset: w = k (+ sign at the fixed coordinate); odd: w = k - neg
      // (k - 1 + neg at the fixed coordinate).
      w[i] = p.odd ? (fix ? p.k[i] - 1 + ng : p.k[i] - ng)
                   : (fix ? p.k[i] + 1 - 2 * ng : p.k[i]);
    }
    uint32_t pc = p.odd ? 1u : 0u;
    int32_t r = (w[0] + w[1] + w[2] + w[3] + w[4] + w[5] + w[6]) & 1;
    int32_t t = (w[7] - r) >> 1;
#pragma unroll
    for (int i = 0; i < 7; ++i) s[i] = 2u * zigzag(w[i]) + pc;
    s[7] = 4u * zigzag(t) + 2u * (uint32_t)r + pc;
  } else if (LAT == 4) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int32_t v[4];
      nearest_d4(y + 4 * h, v);
      int32_t r = (v[0] + v[1] + v[2]) & 1;
      int32_t t = (v[3] - r) >> 1;
      s[4 * h + 0] = zigzag(v[0]);
      s[4 * h + 1] = zigzag(v[1]);
      s[4 * h + 2] = zigzag(v[2]);
      s[4 * h + 3] = 2u * zigzag(t) + (uint32_t)r;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = zigzag(nearest_z(y[i]));
  }
}

// Number of low remainder bits of coordinate c (within its 8-group) fixed by
// membership and not written, for Rice parameter k.
template <int LAT>
__device__ __host__ __forceinline__ constexpr int stripped_low_bits(int c, int k) {
  if (LAT == 8) {
    if (c == 0) return 0;
    if (c == 7) return k < 2 ? k : 2;
    return k < 1 ? k : 1;
  } else if (LAT == 4) {
    return ((c & 3) == 3) ? (k < 1 ? k : 1) : 0;
  }
  return 0;
}

// Restores stripped bits of one 8-group of symbols and returns the lattice
// point; sets *bad when a transmitted copy of a membership bit disagrees.
template <int LAT>
__device__ __forceinline__ void unfold8(uint32_t s[8], int k, int32_t v[8], bool *bad) {
  if (LAT == 8) {
    uint32_t p = s[0] & 1u;
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      if (k >= 1) s[i] |= p;
      else if ((s[i] & 1u) != p) *bad = true;
    }
    int32_t w[8];
    int32_t r = 0;
#pragma unroll
    for (int i = 0; i < 7; ++i) { w[i] = unzigzag(s[i] >> 1); r += w[i]; }
    r &= 1;
    if (k >= 2) s[7] |= (uint32_t)r << 1;
    else if (((s[7] >> 1) & 1u) != (uint32_t)r) *bad = true;
    w[7] = 2 * unzigzag(s[7] >> 2) + r;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 2 * w[i] + (int32_t)p;
  } else if (LAT == 4) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t *q = s + 4 * h;
      int32_t *o = v + 4 * h;
      o[0] = unzigzag(q[0]);
      o[1] = unzigzag(q[1]);
      o[2] = unzigzag(q[2]);
      int32_t r = (o[0] + o[1] + o[2]) & 1;
      if (k >= 1) q[3] |= (uint32_t)r;
      else if ((q[3] & 1u) != (uint32_t)r) *bad = true;
      o[3] = 2 * unzigzag(q[3] >> 1) + r;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = unzigzag(s[i]);
  }
}

// Remainder bits written per tile.
// Remainder bits written per 8 coordinates and per tile.
template <int LAT>
__device__ __host__ __forceinline__ constexpr int rbits8(int k) {
  return 8 * k - stripped_low_bits<LAT>(0, k) - stripped_low_bits<LAT>(1, k) -
         stripped_low_bits<LAT>(2, k) - stripped_low_bits<LAT>(3, k) -
         stripped_low_bits<LAT>(4, k) - stripped_low_bits<LAT>(5, k) -
         stripped_low_bits<LAT>(6, k) - stripped_low_bits<LAT>(7, k);
}
template <int LAT>
__device__ __host__ __forceinline__ constexpr int tile_rbits(int k) {
  return 16 * rbits8<LAT>(k);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint32_t b = __float_as_uint(f);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

}  // namespace hq

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
// CD9E8D57 and Weyl key increments 9E3779B9 and BB67AE85.  Each half-round
// product is one 32x32->64 multiply.
template <class Keys>
__device__ __forceinline__ uint4 philox10(uint4 c, const Keys &key) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)c.x * 0xD2511F53u;
    const uint64_t p1 = (uint64_t)c.z * 0xCD9E8D57u;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ key.k0[r], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ key.k1[r], (uint32_t)p0);
  }
  return c;
}

constexpr uint32_t kDitherTag = 0x44495448u;   // 'DITH'

// The four Philox words of 8-coordinate group j of a tile: coordinate 2m
// takes the low half of word m, coordinate 2m+1 the high half.
template <class Keys>
__device__ __forceinline__ uint4 dither_words(const Keys &key, uint64_t tile, uint32_t j) {
  return philox10(make_uint4((uint32_t)tile, (uint32_t)(tile >> 32), j, kDitherTag), key);
}
// The 16-bit value b in the low / high half of w as an exact float: the two
// bytes moved under the exponent of 2^23 (one byte permute), then 2^23
// subtracted.
__device__ __forceinline__ float half_lo(uint32_t w) {
  return __fsub_rn(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7610)), 8388608.0f);
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __fsub_rn(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7632)), 8388608.0f);
}
// With b as above these give the grid midpoints exactly (at most 17
// significant bits), in one fused multiply-add:
//   -1   + (b + 1/2) 2^-15 = b 2^-15 + (-1 + 2^-16)
//   -2   + (b + 1/2) 2^-14 = b 2^-14 + (-2 + 2^-15)
//   -1/2 + (b + 1/2) 2^-16 = b 2^-16 + (-1/2 + 2^-17)
constexpr float kGrid15 = -1.0f + 0x1p-16f;
constexpr float kGrid14 = -2.0f + 0x1p-15f;
constexpr float kGrid16 = -0.5f + 0x1p-17f;

// ---------------------------------------------------------------- FWHT-128
// Unnormalised Walsh-Hadamard transform, natural (Sylvester) order, stages
// h = 1, 2, ..., 64 in that order, each butterfly (a, b) -> (a + b, a - b)
// rounded once (Method 1): fwht128_t8 below.

// ---------------------------------------------------------------- packed fp32 pairs
// sm_100+ executes add / sub / mul / fma on a pair of fp32 values in one
// instruction; each half rounds to nearest even exactly as the scalar
// instruction does, so a pair operation equals two scalar ones bit for bit.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// (lo, hi) <- (lo + hi, lo - hi) on two pairs: the butterfly of two stages
// positions at once.
__device__ __forceinline__ void bfly2(float &a0, float &a1, float &b0, float &b1) {
  const uint64_t A = pk2(a0, a1), B = pk2(b0, b1);
  upk2(add2(A, B), a0, a1);
  upk2(sub2(A, B), b0, b1);
}

// The transform with a tile spread over 8 consecutive lanes (lane r holds
// coordinates 16r .. 16r+15) and the three cross-lane stages done in
// registers after a transposition through shared memory.  Stages 1, 2, 4 run
// on pairs (x[j], x[j+8]), stage 8 inside those pairs; each pair is stored to
// row j of an 8-row table (coordinate i at row i mod 8, column i / 8, rows
// kTrRow floats apart), lane c reads row c back (coordinates c + 8m,
// m = 0..15) and runs stages 16, 32, 64 on pairs of adjacent columns, then
// writes the row back: the result stays in the table.  Every coordinate goes
// through the additions of the definition above, stage by stage in order,
// whichever lane makes them.  `tile` is the tile's table (kTrTile floats, 16-byte aligned), private
// to its 8 lanes; with rows of 20 floats and tables 176 floats apart, the
// pair stores (16 lanes = two tiles) and the 16-byte row loads and stores
// (8 lanes = one tile) of a warp are free of bank conflicts.  All 32 lanes of
// the warp must call it.
constexpr int kTrRow = 20;
constexpr int kTrTile = 176;
__device__ __forceinline__ void fwht128_t8_smem(float x[16], float *tile, int r) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j & h) continue;
      bfly2(x[j], x[j + 8], x[j + h], x[j + h + 8]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float a = x[j], b = x[j + 8];
    x[j] = __fadd_rn(a, b);
    x[j + 8] = __fsub_rn(a, b);
  }
  // pair (x[j], x[j+8]) = coordinates 16r + j, 16r + j + 8: row j, columns 2r, 2r + 1
  const uint32_t pa = (uint32_t)__cvta_generic_to_shared(tile + 2 * r);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(pa + 4u * kTrRow * j), "f"(x[j]),
                 "f"(x[j + 8])
                 : "memory");
  __syncwarp();
  float y[16];
  const uint32_t row = (uint32_t)__cvta_generic_to_shared(tile + kTrRow * r);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(y[4 * q]), "=f"(y[4 * q + 1]), "=f"(y[4 * q + 2]), "=f"(y[4 * q + 3])
                 : "r"(row + 16u * q)
                 : "memory");
  // y[m] = coordinate r + 8m: stages 16, 32, 64 act on bits 1, 2, 3 of m
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      if (a & h) continue;
      bfly2(y[2 * a], y[2 * a + 1], y[2 * (a + h)], y[2 * (a + h) + 1]);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(row + 16u * q), "f"(y[4 * q]),
                 "f"(y[4 * q + 1]), "f"(y[4 * q + 2]), "f"(y[4 * q + 3])
                 : "memory");
  __syncwarp();
}
// The whole transform back in registers: x[j], x[j + 8] = coordinates 16r + j, 16r + j + 8.
__device__ __forceinline__ void fwht128_t8(float x[16], float *tile, int r) {
  fwht128_t8_smem(x, tile, r);
  const uint32_t pa = (uint32_t)__cvta_generic_to_shared(tile + 2 * r);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(x[j]), "=f"(x[j + 8])
                 : "r"(pa + 4u * kTrRow * j)
                 : "memory");
}

// 1 << n for n < 32, and 0 for n >= 32 (PTX shl clamps the shift amount).
__device__ __forceinline__ uint32_t bit_at(uint32_t n) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(1u), "r"(n));
  return r;
}

// x << n with the PTX rule for n >= 32 (the result is 0), unlike C's shift.
__device__ __forceinline__ uint32_t shl_clamp(uint32_t x, uint32_t n) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(n));
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

// A2 (hexagonal, minimal distance 1) as codes (m, n), m = n mod 2, for the
// point (m / 2, h n): the nearer of the two cosets of Z x sqrt(3) Z, each
// rounded coordinate by coordinate (c = fl32(1/sqrt 3), h = fl32(sqrt(3)/2));
// exact ties go to the coset with m, n even.
constexpr float kA2C = 0x1.279a74p-1f;           // fl32(1/sqrt 3)
constexpr float kA2H = 0x1.bb67aep-1f;           // fl32(sqrt(3)/2)
// int32 -> float for |n| < 2^22 (exact) by the magic number, on the FMA pipe
__device__ __forceinline__ float small_int_to_float(int32_t n) {
  return __fsub_rn(__int_as_float(0x4B400000 + n), kMagic1);
}
__device__ __forceinline__ float a2_px(int32_t m) { return __fmul_rn(0.5f, small_int_to_float(m)); }
__device__ __forceinline__ float a2_py(int32_t n) { return __fmul_rn(kA2H, small_int_to_float(n)); }
__device__ __forceinline__ void nearest_a2(float x, float y, int32_t &m, int32_t &n) {
  const float yc = __fmul_rn(y, kA2C);
  // rint(x), rint(yc), rint(x - 1/2), rint(yc - 1/2) by the magic number
  // (round half to even, exact below 2^22; |x|, |yc| stay below 2^21)
  const float Tx = __fadd_rn(x, kMagic1), Ty = __fadd_rn(yc, kMagic1);
  const float Txo = __fadd_rn(__fsub_rn(x, 0.5f), kMagic1);
  const float Tyo = __fadd_rn(__fsub_rn(yc, 0.5f), kMagic1);
  const float fx = __fsub_rn(Tx, kMagic1), fy = __fsub_rn(Ty, kMagic1);
  const float fxo = __fsub_rn(Txo, kMagic1), fyo = __fsub_rn(Tyo, kMagic1);
  const int32_t me = 2 * (int32_t)(fbits(Tx) - fbits(kMagic1));
  const int32_t ne = 2 * (int32_t)(fbits(Ty) - fbits(kMagic1));
  const int32_t mo = 2 * (int32_t)(fbits(Txo) - fbits(kMagic1)) + 1;
  const int32_t no = 2 * (int32_t)(fbits(Tyo) - fbits(kMagic1)) + 1;
  // the points (m / 2, fl(h n)): m / 2 = rint (even coset) or rint + 1/2
  // (odd coset), n = 2 rint or 2 rint + 1, all exact
  const float dxe = __fsub_rn(x, fx), dye = __fsub_rn(y, __fmul_rn(kA2H, __fadd_rn(fy, fy)));
  const float dxo = __fsub_rn(x, __fadd_rn(fxo, 0.5f));
  const float dyo = __fsub_rn(y, __fmul_rn(kA2H, __fmaf_rn(2.0f, fyo, 1.0f)));
  const float de = __fmaf_rn(dxe, dxe, __fmul_rn(dye, dye));
  const float dd = __fmaf_rn(dxo, dxo, __fmul_rn(dyo, dyo));
  const bool odd = dd < de;
  m = odd ? mo : me;
  n = odd ? no : ne;
}

// ---------------------------------------------------------------- dither
// a * sign(e): the sign bit of e flips a (e is never zero here).
__device__ __forceinline__ float mulsign(float a, float e) {
  return __uint_as_float(__float_as_uint(a) ^ (__float_as_uint(e) & 0x80000000u));
}

// U ~ Uniform(V(Lambda)) for the 8 coordinates of group j of a tile (Method 4):
// a grid point u0 of a box that tiles space by the lattice, minus Q(u0).
// The boxes are centred, so Q(u0) needs the general rounding on one
// coordinate per vector only; the rest of the nearest-point rule is the same
// as in quantize_fold16_e8 / nearest_d4 (largest-error / smallest-error
// coordinate, first index among equals, the odd E8 coset only when strictly
// nearer).
template <int LAT, class Keys>
__device__ __forceinline__ void dither8(const Keys &key, uint64_t tile, uint32_t j, float u[8]) {
  const uint4 w4 = dither_words(key, tile, j);
  const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
  if (LAT == 8) {
    float e[8];
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      e[2 * m] = __fmaf_rn(half_lo(w[m]), 0x1p-15f, kGrid15);
      e[2 * m + 1] = __fmaf_rn(half_hi(w[m]), 0x1p-15f, kGrid15);
    }
    e[6] = __fmaf_rn(half_lo(w[3]), 0x1p-15f, kGrid15);
    const float u07 = __fmaf_rn(half_hi(w[3]), 0x1p-14f, kGrid14);   // in (-2, 2)
    // coordinates 0..6 lie in (-1, 1): nearest even integer 0, error = u0
    const float T7 = __fadd_rn(u07, kMagic2);
    const float F7 = __fsub_rn(T7, kMagic2);
    e[7] = __fsub_rn(u07, F7);
    uint32_t sx = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) sx ^= __float_as_uint(e[i]);
    const uint32_t pA = __float_as_uint(T7) & 1u;          // parity of F7 / 2
    const uint32_t pB = pA ^ (sx >> 31);
    float S = fabsf(e[0]), mx = fabsf(e[0]), mn = fabsf(e[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      const float ai = fabsf(e[i]);
      S = __fadd_rn(S, ai);
      mx = fmaxf(mx, ai);
      mn = fminf(mn, ai);
    }
    float D = __fmaf_rn(-2.0f, S, pA ? 4.0f : 8.0f);
    if (pB) D = __fmaf_rn(4.0f, mn, D);
    if (pA) D = __fmaf_rn(4.0f, mx, D);
    const bool odd = D < 0.0f;
    const float m = odd ? mn : mx;
    bool open = odd ? (pB != 0u) : (pA != 0u);   // a parity fix is still to place
    const float wb = odd ? 1.0f : 0.0f, wh = odd ? -1.0f : 2.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool hit = open && fabsf(e[i]) == m;
      open = open && !hit;
      u[i] = __fsub_rn(e[i], mulsign(hit ? wh : wb, e[i]));
    }
  } else if (LAT == 4) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float e[4];
      e[0] = __fmaf_rn(half_lo(w[2 * h]), 0x1p-16f, kGrid16);
      e[1] = __fmaf_rn(half_hi(w[2 * h]), 0x1p-16f, kGrid16);
      e[2] = __fmaf_rn(half_lo(w[2 * h + 1]), 0x1p-16f, kGrid16);
      const float u03 = __fmaf_rn(half_hi(w[2 * h + 1]), 0x1p-15f, kGrid15);   // in (-1, 1)
      const float T3 = __fadd_rn(u03, kMagic1);
      e[3] = __fsub_rn(u03, __fsub_rn(T3, kMagic1));
      bool open = (__float_as_uint(T3) & 1u) != 0u;   // odd sum: move the worst coordinate
      const float mx = fmaxf(fmaxf(fabsf(e[0]), fabsf(e[1])), fmaxf(fabsf(e[2]), fabsf(e[3])));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool hit = open && fabsf(e[i]) == mx;
        open = open && !hit;
        u[4 * h + i] = hit ? __fsub_rn(e[i], mulsign(1.0f, e[i])) : e[i];
      }
    }
  } else if (LAT == 2) {
    // pair m: u0 = (-1/2 + (b + 1/2) 2^-16, fl(h (-1 + (b' + 1/2) 2^-15))) on
    // the box [-1/2, 1/2) x [-h, h), two cells of A2; u = u0 - point(Q(u0))
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float x0 = __fmaf_rn(half_lo(w[m]), 0x1p-16f, kGrid16);
      const float y0 = __fmul_rn(kA2H, __fmaf_rn(half_hi(w[m]), 0x1p-15f, kGrid15));
      int32_t qm, qn;
      nearest_a2(x0, y0, qm, qn);
      u[2 * m] = __fsub_rn(x0, a2_px(qm));
      u[2 * m + 1] = __fsub_rn(y0, a2_py(qn));
    }
  } else {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      u[2 * m] = __fmaf_rn(half_lo(w[m]), 0x1p-16f, kGrid16);
      u[2 * m + 1] = __fmaf_rn(half_hi(w[m]), 0x1p-16f, kGrid16);
    }
  }
}

// ---------------------------------------------------------------- fold / strip
// Nearest point and symbols of one 8-coordinate group (Method 2 and 3) for
// D4, A2 and Z (E8: quantize_fold16_e8).  D4 (two vectors):
// r = parity(v0+v1+v2), t = (v3 - r)/2, s_3 = 2Z(t) + r; A2 (four pairs):
// s_0 = Z(n), s_1 = 2Z((m - p)/2) + p with p = n mod 2; Z: s = Z(v).
template <int LAT>
__device__ __forceinline__ void quantize_fold8(const float y[8], uint32_t s[8]) {
  static_assert(LAT != 8, "E8 codes both 8-vectors of a lane at once: quantize_fold16_e8");
  if (LAT == 4) {
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
  } else if (LAT == 2) {
    // pair (m, n): p = n mod 2, w = (m - p)/2; s_0 = Z(n), s_1 = 2 Z(w) + p
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      int32_t m, n;
      nearest_a2(y[2 * h], y[2 * h + 1], m, n);
      const int32_t p = n & 1;
      s[2 * h] = zigzag(n);
      s[2 * h + 1] = 2u * zigzag((m - p) >> 1) + (uint32_t)p;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = zigzag(nearest_z(y[i]));
  }
}

// Nearest point of 2E8 and the Rice symbols of the lane's two 8-vectors
// (Method 2 and 3; y[i] and y[8 + i] are coordinate i of each).  Per vector:
// F_i = y_i rounded to the nearest even integer (magic-number rounding),
// e_i = y_i - F_i (exact).  The even coset's nearest point is F, with the
// coordinate of largest |e_i| moved by 2 sign(e_i) when sum F_i / 2 is odd;
// the odd coset's is F + sign(e), with the coordinate of smallest |e_i| moved
// back (-sign) when its parity needs it (an error of -0 counts as negative,
// the first index among equal |e_i| moves).  The odd coset wins only when
// the exact difference of the two squared distances, (8 - 4pA) - 2 sum|e| +
// 4pB min|e| + 4pA max|e|, evaluated in fp32 in that order, is negative.
// Fold (p = coset): s_i = 2Z(w_i) + p with w_i = (v_i - p)/2, i.e.
// |2 v_i + 1 - 2p| - 1 + p (exact in fp32), for i < 7; r = parity of
// w_0 + .. + w_6, s_7 = 4Z((w_7 - r)/2) + 2r + p.  The roundings, errors,
// lattice point and fold run on fp32 pairs (one vector per half); the
// per-vector decision in scalar code.
__device__ __forceinline__ void quantize_fold16_e8(const float y[16], uint32_t s[16]) {
  float F[16], e[16];
  const uint64_t M2 = pk2(kMagic2, kMagic2);
  uint64_t SF = 0, PE = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t Y = pk2(y[i], y[8 + i]);
    const uint64_t FF = sub2(add2(Y, M2), M2);
    const uint64_t E = sub2(Y, FF);
    upk2(E, e[i], e[8 + i]);
    upk2(FF, F[i], F[8 + i]);
    SF = i == 0 ? FF : add2(SF, FF);             // sum F (exact: even integers, |F| <= 2^20 + 2)
    PE = i == 0 ? E : mul2(PE, E);               // its sign = the XOR of the errors' signs
  }
  // parity of sum F / 2 from the magic-number rounding of the exact half sum;
  // the sign parity of the errors from their product (the sign of a product
  // is the XOR of the factors' signs, zeros included, whatever the rounding)
  uint32_t par[2], sx[2];
  {
    float h0, h1, p0, p1;
    upk2(fma2(SF, pk2(0.5f, 0.5f), pk2(kMagic1, kMagic1)), h0, h1);
    upk2(PE, p0, p1);
    par[0] = __float_as_uint(h0);
    par[1] = __float_as_uint(h1);
    sx[0] = __float_as_uint(p0);
    sx[1] = __float_as_uint(p1);
  }
  float c[16];
  bool odd[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float *eh = e + 8 * h;
    const uint32_t pA = par[h] & 1u, pB = pA ^ (sx[h] >> 31);
    float S = fabsf(eh[0]), mx = fabsf(eh[0]), mn = fabsf(eh[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      const float ai = fabsf(eh[i]);
      S = __fadd_rn(S, ai);
      mx = fmaxf(mx, ai);
      mn = fminf(mn, ai);
    }
    float D = __fmaf_rn(-2.0f, S, pA ? 4.0f : 8.0f);
    if (pB) D = __fmaf_rn(4.0f, mn, D);
    if (pA) D = __fmaf_rn(4.0f, mx, D);
    odd[h] = D < 0.0f;
    const float m = odd[h] ? mn : mx;
    bool open = odd[h] ? (pB != 0u) : (pA != 0u);
    const float wb = odd[h] ? 1.0f : 0.0f, wh = odd[h] ? -1.0f : 2.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool hit = open && fabsf(eh[i]) == m;
      open = open && !hit;
      c[8 * h + i] = __uint_as_float(__float_as_uint(hit ? wh : wb) ^
                                     (__float_as_uint(eh[i]) & 0x80000000u));
    }
  }
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) upk2(add2(pk2(F[i], F[8 + i]), pk2(c[i], c[8 + i])), v[i], v[8 + i]);
  // fold
  uint64_t sum7 = pk2(v[0], v[8]);
#pragma unroll
  for (int i = 1; i < 7; ++i) sum7 = add2(sum7, pk2(v[i], v[8 + i]));
  const uint64_t half = fma2(sum7, pk2(0.5f, 0.5f), pk2(odd[0] ? -3.5f : 0.0f, odd[1] ? -3.5f : 0.0f));
  float hr0, hr1;
  upk2(add2(half, pk2(kMagic1, kMagic1)), hr0, hr1);
  const uint32_t r0 = __float_as_uint(hr0) & 1u, r1 = __float_as_uint(hr1) & 1u;
  const uint64_t C1 = pk2(odd[0] ? -1.0f : 1.0f, odd[1] ? -1.0f : 1.0f);
  const float cs0 = odd[0] ? kMagic1 : kMagic1 - 1.0f, cs1 = odd[1] ? kMagic1 : kMagic1 - 1.0f;
  const uint64_t TWO = pk2(2.0f, 2.0f);
#pragma unroll
  for (int i = 0; i < 7; ++i) {
    float a0, a1;
    upk2(fma2(TWO, pk2(v[i], v[8 + i]), C1), a0, a1);
    s[i] = __float_as_uint(__fadd_rn(fabsf(a0), cs0)) - 0x4B400000u;
    s[8 + i] = __float_as_uint(__fadd_rn(fabsf(a1), cs1)) - 0x4B400000u;
  }
  const float p0 = odd[0] ? 1.0f : 0.0f, p1 = odd[1] ? 1.0f : 0.0f;
  const float rf0 = r0 ? 1.0f : 0.0f, rf1 = r1 ? 1.0f : 0.0f;
  float a0, a1;
  upk2(fma2(TWO, pk2(v[7], v[15]),
            fma2(pk2(-4.0f, -4.0f), pk2(rf0, rf1), pk2(2.0f - 2.0f * p0, 2.0f - 2.0f * p1))),
       a0, a1);
  float b0, b1;
  upk2(fma2(TWO, pk2(rf0, rf1), pk2(p0 - 2.0f + kMagic1, p1 - 2.0f + kMagic1)), b0, b1);
  s[7] = __float_as_uint(__fadd_rn(fabsf(a0), b0)) - 0x4B400000u;
  s[15] = __float_as_uint(__fadd_rn(fabsf(a1), b1)) - 0x4B400000u;
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
  } else if (LAT == 2) {
    return (c & 1) ? (k < 1 ? k : 1) : 0;
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
  } else if (LAT == 2) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int32_t n = unzigzag(s[2 * h]);
      const uint32_t p = (uint32_t)n & 1u;
      uint32_t s1 = s[2 * h + 1];
      if (k >= 1) s1 |= p;
      else if ((s1 & 1u) != p) *bad = true;
      v[2 * h] = 2 * unzigzag(s1 >> 1) + (int32_t)p;
      v[2 * h + 1] = n;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = unzigzag(s[i]);
  }
}

// Lattice point of 8 codes: the identity for Z, D4 and 2E8 (exact int ->
// float for |v| < 2^22 by the magic-number conversion); for A2 each pair
// (m, n) is (m / 2, fl(h n)).
template <int LAT>
__device__ __forceinline__ void point8(const int32_t v[8], float fv[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (LAT == 2) fv[i] = (i & 1) ? a2_py(v[i]) : a2_px(v[i]);
    else fv[i] = __fsub_rn(__int_as_float(0x4B400000 + v[i]), kMagic1);
  }
}

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

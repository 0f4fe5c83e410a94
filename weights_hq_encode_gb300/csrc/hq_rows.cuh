// hq_rows.cuh -- rotation of query and activation rows into the lattice
// domain, x' = s_dec * H * D * (R) x per 128-dimension tile (HyperQuant
// summary, Method 1, applied to the other operand of the fused products).
//
// A row is spread over 8 consecutive lanes like a codec tile (lane r holds
// dimensions 16 r .. 16 r + 15), so the transform is the tiled one.  The
// optional dense rotation is one fused multiply-add chain over j = 0..127
// from +0 per output, the sign flips are exact and the transform rounds each
// butterfly once, stage by stage in order, as its definition states.
#pragma once
#include <cuda_runtime.h>

#include "hq_device.cuh"

namespace hq {

// Lane r of a row: src = the row's 128 bf16 values (nullptr: a padding row,
// read as zeros and not stored), vec = src may be read 16 bytes at a time,
// R = the row's 128 x 128 rotation (row-major, 16-byte aligned) or nullptr,
// mw = the 16 sign bits of dimensions 16 r .. 16 r + 15 (bit i: dimension
// 16 r + i), dst = the row's 128 fp32 outputs (16-byte aligned), tile = the
// row's kTrTile-float table in shared memory (16-byte aligned, private to
// its 8 lanes).  All 32 lanes of the warp must call it.
__device__ __forceinline__ void rotate_row_t8(const uint16_t *src, bool vec, const float *R,
                                              uint32_t mw, float s_dec, float *dst, float *tile,
                                              int r) {
  float x[16];
  {
    uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (src != nullptr) {
      const uint16_t *q = src + 16 * r;
      if (vec) {
        const uint4 v0 = __ldg(reinterpret_cast<const uint4 *>(q));
        const uint4 v1 = __ldg(reinterpret_cast<const uint4 *>(q) + 1);
        w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
        w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = (uint32_t)q[2 * i] | ((uint32_t)q[2 * i + 1] << 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {               // bf16 -> fp32 is exact
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  if (R != nullptr) {                            // x <- R x, the inputs staged in the table
    float4 *xs = reinterpret_cast<float4 *>(tile + 16 * r);
#pragma unroll
    for (int c = 0; c < 4; ++c) xs[c] = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
    __syncwarp();
    const float4 *xin = reinterpret_cast<const float4 *>(tile);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 *Ri = reinterpret_cast<const float4 *>(R + (int64_t)(16 * r + i) * kTile);
      float acc = 0.0f;
#pragma unroll 8
      for (int j4 = 0; j4 < kTile / 4; ++j4) {
        const float4 rv = __ldg(Ri + j4), xv = xin[j4];
        acc = __fmaf_rn(rv.x, xv.x, acc);
        acc = __fmaf_rn(rv.y, xv.y, acc);
        acc = __fmaf_rn(rv.z, xv.z, acc);
        acc = __fmaf_rn(rv.w, xv.w, acc);
      }
      x[i] = acc;
    }
    __syncwarp();                                // all inputs read: the transform reuses the table
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(__float_as_uint(x[i]) ^ (((mw >> i) & 1u) << 31));
  fwht128_t8(x, tile, r);
  if (src == nullptr) return;
  float4 *o = reinterpret_cast<float4 *>(dst + 16 * r);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    o[c] = make_float4(__fmul_rn(x[4 * c], s_dec), __fmul_rn(x[4 * c + 1], s_dec),
                       __fmul_rn(x[4 * c + 2], s_dec), __fmul_rn(x[4 * c + 3], s_dec));
}

// Rows handled by one block of the rotation kernels (8 lanes a row).
constexpr int kRowThreads = 256;

}  // namespace hq

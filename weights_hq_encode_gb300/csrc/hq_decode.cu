// hq_decode.cu -- decoder and fused score kernel of the HyperQuant tile codec.
//
// One warp per index group of 32 tiles, one lane per tile.  The warp finds
// the start of every tile's unary section by a popcount scan of the group's
// U-area (every one bit there terminates a symbol, 128 per tile), then each
// lane reads its remainders at their fixed position, its unary codes with
// count-leading-zeros, restores the stripped bits, regenerates the dither and
// inverts the transform (HyperQuant summary, Method 1-4 in reverse).  Every
// loop is bounded by the group's own word count from the index, and a group
// that fails any check is written as zeros with HQ_ERR_CORRUPT.
//
// hq_decode_qk (the summary's closing section, fused decode + MMA) decodes K
// tiles only to the lattice domain e = v - u and dots them with queries that
// were rotated once into the same domain, q' = s_dec H D q, so K is never
// written and no inverse transform is run per key.
#include <cuda_runtime.h>

#include "hq_device.cuh"
#include "hq_internal.h"

namespace hq {

constexpr int kDecThreads = 128;
constexpr int kDecGroups = kDecThreads / 32;

__device__ __forceinline__ uint32_t get_bits(const uint32_t *p, uint64_t pos, int nb) {
  uint64_t w = pos >> 5;
  int sh = (int)(pos & 31);
  uint32_t hi = __ldg(p + w);
  uint32_t lo = (sh + nb > 32) ? __ldg(p + w + 1) : 0u;
  return __funnelshift_l(lo, hi, sh) >> (32 - nb);
}

// MSB-first position (0..31) of the n-th (1-based) set bit of x.
__device__ __forceinline__ int nth_set_bit_msb(uint32_t x, int n) {
  for (int i = 1; i < n; ++i) x &= ~(0x80000000u >> __clz(x));
  return __clz(x);
}

// Decodes the tile of this lane to the lattice-domain values e = v - u.
// Returns false (for the whole warp) when the group is corrupt.
template <int LAT>
__device__ bool decode_group_lane(const DecodeArgs &a, int64_t g, int lane, float e[128],
                                  uint64_t (*s_start)[kGroupTiles + 1]) {
  const int64_t t0 = g * kGroupTiles;
  const int nt = (int)min((int64_t)kGroupTiles, a.n_tiles - t0);
  const uint64_t base = a.offsets[g], end = a.offsets[g + 1];
  const int k = a.rice_k;
  const uint64_t R = (uint64_t)a.rbits;
  bool bad = end < base || end > a.stream_words;
  const uint64_t nwords = bad ? 0 : end - base;
  const uint64_t nbits = nwords * 32;
  const uint64_t ustart = (uint64_t)nt * R;
  if (ustart > nbits) bad = true;
  const uint32_t *p = a.stream + base;
  uint64_t *starts = s_start[threadIdx.x >> 5];

  // ---- tile boundaries: popcount scan of the U-area
  uint64_t ones = 0, uend = 0;
  const uint64_t want = 128ull * (uint64_t)nt;
  if (!bad) {
    if (lane == 0) starts[0] = ustart;
    for (uint64_t wb = ustart >> 5; wb < nwords; wb += 32) {
      uint64_t w = wb + lane;
      uint32_t word = w < nwords ? __ldg(p + w) : 0u;
      if (w == (ustart >> 5)) word &= 0xFFFFFFFFu >> (ustart & 31);
      uint32_t pc = __popc(word);
      uint32_t incl = pc;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      uint64_t before = ones + incl - pc;
      uint64_t m = (before / 128 + 1) * 128;       // next tile boundary (in ones)
      if (pc && m <= before + pc && m <= want) {
        int pos = nth_set_bit_msb(word, (int)(m - before));
        uint64_t bit = w * 32 + (uint64_t)pos + 1;
        int ti = (int)(m / 128);
        if (ti < nt) starts[ti] = bit;
        else uend = bit;
      }
      ones += __shfl_sync(0xffffffffu, incl, 31);
    }
    // the lane that found the end of the last tile shares it
    uint64_t ue = uend;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) ue = max(ue, __shfl_xor_sync(0xffffffffu, ue, d));
    uend = ue;
    if (ones != want || ((uend + 31) >> 5) != nwords) bad = true;
  }
  __syncwarp();

  // ---- per-lane parse
  uint32_t sym[128];
  bool lbad = false;
  if (!bad && lane < nt) {
    if (R > 0) {
      uint64_t pos = (uint64_t)lane * R;
#pragma unroll
      for (int j = 0; j < 128; ++j) {
        int lowb = stripped_low_bits<LAT>(j & 7, k);
        int nb = k - lowb;
        sym[j] = nb > 0 ? (get_bits(p, pos, nb) << lowb) : 0u;
        pos += (uint64_t)max(nb, 0);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 128; ++j) sym[j] = 0u;
    }
    uint64_t pos = starts[lane];
    const uint64_t stop = (lane + 1 < nt) ? starts[lane + 1] : uend;
    const uint32_t qmax = (kSymbolLimit - 1u) >> k;
#pragma unroll
    for (int j = 0; j < 128; ++j) {
      uint32_t q = 0;
      bool done = lbad;
      while (!done) {
        if (pos >= stop) { lbad = true; break; }
        uint32_t x = __ldg(p + (pos >> 5)) << (pos & 31);
        uint32_t avail = 32u - (uint32_t)(pos & 31);
        if (x) {
          uint32_t z = __clz(x);
          q += z;
          pos += z + 1;
          done = true;
        } else {
          q += avail;
          pos += avail;
          if (q > qmax) { lbad = true; break; }
        }
      }
      if (q > qmax) lbad = true;
      sym[j] |= q << k;
    }
    if (!lbad && pos != stop) lbad = true;
  }
  // ---- unfold, dither, e = v - u
  if (!bad && !lbad && lane < nt) {
    const uint64_t gt = a.tile_base + (uint64_t)(t0 + lane);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      int32_t v[8];
      unfold8<LAT>(sym + 8 * j, k, v, &lbad);
      float u[8];
      if (a.dither) {
        dither8<LAT>(a.dither_seed, gt, (uint32_t)j, u);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) u[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) e[8 * j + i] = __fsub_rn((float)v[i], u[i]);
    }
  }
  bad = bad || __any_sync(0xffffffffu, lbad);
  return !bad;
}

template <int LAT>
__global__ void __launch_bounds__(kDecThreads)
decode_kernel(DecodeArgs a) {
  __shared__ uint64_t s_start[kDecGroups][kGroupTiles + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t g = (int64_t)blockIdx.x * kDecGroups + warp;
  if (g >= a.n_groups) return;
  float e[128];
  bool ok = decode_group_lane<LAT>(a, g, lane, e, s_start);
  const int64_t t = g * kGroupTiles + lane;
  if (t >= a.n_tiles) return;
  if (!ok) {
    if (lane == 0) atomicOr(a.status, (uint32_t)HQ_ERR_CORRUPT);
#pragma unroll
    for (int i = 0; i < 128; ++i) e[i] = 0.0f;
  } else {
    fwht128(e);
    const uint32_t *mask = a.signs + 4 * (t / a.tiles_per_segment);
    uint32_t m[4] = {__ldg(mask), __ldg(mask + 1), __ldg(mask + 2), __ldg(mask + 3)};
#pragma unroll
    for (int i = 0; i < 128; ++i) {
      float r = __fmul_rn(e[i], a.s_dec);
      e[i] = ((m[i >> 5] >> (i & 31)) & 1u) ? -r : r;
    }
  }
  if (a.out_kind == HQ_OUT_F32) {
    float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) + t * kTile);
#pragma unroll
    for (int c = 0; c < 32; ++c) dst[c] = make_float4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
  } else {
    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.out) + t * kTile);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h)
        w[h] = (uint32_t)f32_to_bf16_rn(e[8 * c + 2 * h]) |
               ((uint32_t)f32_to_bf16_rn(e[8 * c + 2 * h + 1]) << 16);
      dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// q'[row] = s_dec * H * (D_h q[row]) for row = b * Hq + hq, h = hq / (Hq / n_kv).
__global__ void rotate_queries_kernel(QkArgs a) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= a.B * a.Hq) return;
  const int hq = row % a.Hq, h = hq / (a.Hq / a.n_kv);
  const int64_t seg = ((int64_t)h * a.n_tokens) / a.dec.tiles_per_segment;
  const uint32_t *mask = a.dec.signs + 4 * seg;
  float x[128];
  const uint16_t *q = a.q + (int64_t)row * kTile;
#pragma unroll
  for (int i = 0; i < 128; ++i) {
    float f = __uint_as_float((uint32_t)q[i] << 16);
    x[i] = ((mask[i >> 5] >> (i & 31)) & 1u) ? -f : f;
  }
  fwht128(x);
#pragma unroll
  for (int i = 0; i < 128; ++i) a.qrot[(int64_t)row * kTile + i] = __fmul_rn(x[i], a.dec.s_dec);
}

template <int LAT>
__global__ void __launch_bounds__(kDecThreads)
scores_kernel(QkArgs a) {
  __shared__ uint64_t s_start[kDecGroups][kGroupTiles + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t g = (int64_t)blockIdx.x * kDecGroups + warp;
  if (g >= a.dec.n_groups) return;
  float e[128];
  bool ok = decode_group_lane<LAT>(a.dec, g, lane, e, s_start);
  const int64_t tile = g * kGroupTiles + lane;
  if (tile >= a.dec.n_tiles) return;
  if (!ok) {
    if (lane == 0) atomicOr(a.dec.status, (uint32_t)HQ_ERR_CORRUPT);
#pragma unroll
    for (int i = 0; i < 128; ++i) e[i] = 0.0f;
  }
  const int h = (int)(tile / a.n_tokens);
  const int64_t tok = tile - (int64_t)h * a.n_tokens;
  const int G = a.Hq / a.n_kv;
  for (int b = 0; b < a.B; ++b) {
    for (int gq = 0; gq < G; ++gq) {
      const int64_t row = (int64_t)b * a.Hq + (int64_t)h * G + gq;
      const float4 *qr = reinterpret_cast<const float4 *>(a.qrot + row * kTile);
      float acc = 0.0f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float4 v = __ldg(qr + c);
        acc = __fmaf_rn(v.x, e[4 * c], acc);
        acc = __fmaf_rn(v.y, e[4 * c + 1], acc);
        acc = __fmaf_rn(v.z, e[4 * c + 2], acc);
        acc = __fmaf_rn(v.w, e[4 * c + 3], acc);
      }
      a.scores[row * a.n_tokens + tok] = acc;
    }
  }
}

int launch_decode(const DecodeArgs &a, int lattice, cudaStream_t st) {
  dim3 grid((unsigned)((a.n_groups + kDecGroups - 1) / kDecGroups)), block(kDecThreads);
  switch (lattice) {
    case 8: decode_kernel<8><<<grid, block, 0, st>>>(a); break;
    case 4: decode_kernel<4><<<grid, block, 0, st>>>(a); break;
    default: decode_kernel<1><<<grid, block, 0, st>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_decode_qk(const QkArgs &a, int lattice, cudaStream_t st) {
  const int rows = a.B * a.Hq;
  rotate_queries_kernel<<<(rows + 127) / 128, 128, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return 1;
  dim3 grid((unsigned)((a.dec.n_groups + kDecGroups - 1) / kDecGroups)), block(kDecThreads);
  switch (lattice) {
    case 8: scores_kernel<8><<<grid, block, 0, st>>>(a); break;
    case 4: scores_kernel<4><<<grid, block, 0, st>>>(a); break;
    default: scores_kernel<1><<<grid, block, 0, st>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace hq

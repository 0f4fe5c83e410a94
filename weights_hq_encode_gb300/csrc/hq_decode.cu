// hq_decode.cu -- decoder of the HyperQuant tile codec.
//
// One block of 256 threads per index group of 32 tiles: decode_lane (the
// shared decoding step) gives each lane e = v - u for its 16 coordinates;
// the block then inverts the transform (FWHT, x (D s_dec), optional dense
// rotation R^T) and stores contiguous 32-byte (bf16) / 64-byte (fp32) writes
// per lane.  A group that fails any check is written as zeros with
// HQ_ERR_CORRUPT: without the rotation each lane stores what it decoded and
// the block's verdict, taken after the stores, has every lane of a corrupt
// group overwrite its values with zeros (so no block barrier waits for the
// slowest lane's parse before the transform).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hq_decode_lane.cuh"

namespace hq {

// ROT: the dense-rotation variant (an instance of its own, 4 blocks per SM
// with the registers of its 4 x 4 product tile; runtime k only).
template <int LAT, int K, bool ROT>
__global__ void __launch_bounds__(kDecThreads, ROT ? 4 : 8)
decode_kernel(DecodeArgs a) {
  __shared__ uint64_t s_start[kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[2][kDecThreads / 32];
  // D_i * s_dec of the block's first segment, coordinates 16r + j and 16r + j + 8
  // side by side (the pairs a lane holds after the transform); lane r's block
  // c (j = 2c, 2c + 1) at 8c + r, so the 8 lanes of a tile read 128
  // contiguous bytes
  __shared__ float4 s_scale[kTile / 4];
  __shared__ __align__(16) float s_tr[kGroupTiles * kTrTile];  // transposes of the transform
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7;
  const int64_t g = blockIdx.x;
  const int64_t seg0 = div_by(g * kGroupTiles, a.tiles_per_segment, a.seg_shift);
  if (tid < kTile) {
    const uint32_t mword = __ldg(a.signs + 4 * seg0 + (tid >> 5));
    reinterpret_cast<float *>(s_scale)[32 * ((tid & 7) >> 1) + 4 * (tid >> 4) + 2 * (tid & 1) +
                                       ((tid >> 3) & 1)] =
        __uint_as_float(__float_as_uint(a.s_dec) ^ (((mword >> (tid & 31)) & 1u) << 31));
  }
  constexpr int kRS = kTile + 4;                 // row stride of the rotation's operand
  extern __shared__ __align__(16) float s_dyn[];  // ROT: y [32][kRS]
  float e[16];
  // ok: the group's verdict with the rotation, this lane's own without it
  const bool ok = decode_lane<LAT, K, BlockBar, !ROT>(a, g, e, s_start, s_warp);
  const int64_t t = g * kGroupTiles + tl;
  if (ROT && !ok && tid == 0) atomicOr(a.status, (uint32_t)HQ_ERR_CORRUPT);
  // the transform runs on every lane of the block (its transposes synchronise whole warps)
  fwht128_t8(e, s_tr + tl * kTrTile, r);
  const bool tvalid = t < a.n_tiles;
  if (ok && tvalid) {
    // x = D fl(z s_dec) = fl(z (D s_dec)): the sign commutes with rounding
    if (div_by(t, a.tiles_per_segment, a.seg_shift) == seg0) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 sc = s_scale[8 * c + r];
        upk2(mul2(pk2(e[2 * c], e[2 * c + 8]), pk2(sc.x, sc.y)), e[2 * c], e[2 * c + 8]);
        upk2(mul2(pk2(e[2 * c + 1], e[2 * c + 9]), pk2(sc.z, sc.w)), e[2 * c + 1], e[2 * c + 9]);
      }
    } else {
      const uint32_t *mask = a.signs + 4 * (div_by(t, a.tiles_per_segment, a.seg_shift));
      const uint32_t mw = __ldg(mask + (r >> 1)) >> (16 * (r & 1));
#pragma unroll
      for (int i = 0; i < 16; ++i)
        e[i] = __fmul_rn(e[i], __uint_as_float(__float_as_uint(a.s_dec) ^ (((mw >> i) & 1u) << 31)));
    }
  }
  if constexpr (ROT) {                           // x_hat = R^T y, chains over i
    // [32 tiles x 128] x [128 x 128]: y row-major [32][132] in shared memory
    // (later reused for the result), the segment's R row-major through L1
    // (every block of the segment reads the same 64 KB)
    float *s_y = s_dyn;
    const float *Rg = a.rot + seg0 * (int64_t)(kTile * kTile);
    float4 *dy = reinterpret_cast<float4 *>(s_y + tl * kRS + 16 * r);
#pragma unroll
    for (int c = 0; c < 4; ++c) dy[c] = make_float4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
    __syncthreads();
    // thread (tg, oh, l16): tiles 4 tg .. 4 tg + 3 x outputs 64 oh + 4 l16 .. +3,
    // each one fma chain over i = 0..127 from +0
    const int tg = (tid >> 4) & 7, ob = 64 * (tid >> 7) + 4 * (tid & 15);
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[u][c] = 0.0f;
#pragma unroll 2
    for (int i = 0; i < kTile; i += 4) {
      float4 yv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        yv[u] = *reinterpret_cast<const float4 *>(s_y + (4 * tg + u) * kRS + i);
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const float4 rr = __ldg(reinterpret_cast<const float4 *>(Rg + (i + ii) * kTile + ob));
        const float rs[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float yu = ii == 0 ? yv[u].x : ii == 1 ? yv[u].y : ii == 2 ? yv[u].z : yv[u].w;
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[u][c] = __fmaf_rn(rs[c], yu, acc[u][c]);
        }
      }
    }
    __syncthreads();                             // the y area becomes the result area
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<float4 *>(s_y + (4 * tg + u) * kRS + ob) =
          make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 q = *reinterpret_cast<const float4 *>(s_y + tl * kRS + 16 * r + 4 * c);
      e[4 * c] = q.x;
      e[4 * c + 1] = q.y;
      e[4 * c + 2] = q.z;
      e[4 * c + 3] = q.w;
    }
    if (!tvalid) return;
  }
  if (tvalid) {
    if (a.out_kind == HQ_OUT_F32) {
      float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) + t * kTile + 16 * r);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        dst[c] = make_float4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
    } else {
      uint32_t w[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(e[2 * h], e[2 * h + 1]);   // RNE
        w[h] = *reinterpret_cast<const uint32_t *>(&b2);
      }
      uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.out) + t * kTile + 16 * r);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
  if constexpr (!ROT) {
    // every thread of the block reaches this barrier (none has returned)
    if (__syncthreads_or(ok ? 0 : 1)) {
      if (tid == 0) atomicOr(a.status, (uint32_t)HQ_ERR_CORRUPT);
      if (tvalid) {                              // the same bytes, now zeros
        const int n16 = a.out_kind == HQ_OUT_F32 ? 4 : 2;
        uint4 *dst = reinterpret_cast<uint4 *>(a.out) + (t * kTile + 16 * r) / 16 * n16;
        for (int c = 0; c < n16; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

constexpr size_t kDecRotSmemBytes = (size_t)(kGroupTiles * (kTile + 4)) * 4;

template <int LAT, int K, bool ROT = false>
static void launch_dec_one(const DecodeArgs &a, cudaStream_t st) {
  const size_t dyn = ROT ? kDecRotSmemBytes : 0;
  if (dyn)
    cudaFuncSetAttribute(decode_kernel<LAT, K, ROT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)dyn);
  decode_kernel<LAT, K, ROT><<<dim3((unsigned)a.n_groups), dim3(kDecThreads), dyn, st>>>(a);
}

template <int LAT>
static void launch_dec_lat(const DecodeArgs &a, cudaStream_t st) {
  if (a.rot != nullptr) {                        // the rotation variant takes k at run time
    launch_dec_one<LAT, -1, true>(a, st);
    return;
  }
  switch (a.rice_k) {
    case 0: launch_dec_one<LAT, 0>(a, st); break;
    case 1: launch_dec_one<LAT, 1>(a, st); break;
    case 2: launch_dec_one<LAT, 2>(a, st); break;
    case 3: launch_dec_one<LAT, 3>(a, st); break;
    case 4: launch_dec_one<LAT, 4>(a, st); break;
    case 5: launch_dec_one<LAT, 5>(a, st); break;
    case 6: launch_dec_one<LAT, 6>(a, st); break;
    case 7: launch_dec_one<LAT, 7>(a, st); break;
    case 8: launch_dec_one<LAT, 8>(a, st); break;
    default: launch_dec_one<LAT, -1>(a, st); break;
  }
}

int launch_decode(const DecodeArgs &a, int lattice, cudaStream_t st) {
  switch (lattice) {
    case 8: launch_dec_lat<8>(a, st); break;
    case 4: launch_dec_lat<4>(a, st); break;
    case 2: launch_dec_lat<2>(a, st); break;
    default: launch_dec_lat<1>(a, st); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace hq

// hq_fused_gemm.cu -- products with compressed weights (hq_decode_gemm), the
// summary's closing section, fused decode + MMA: the activations are rotated
// once into the lattice domain (x' = s_dec H D R x per 128-column tile), each
// weight tile is decoded only to e = v - u and dotted with its slice of x',
// and the tiles' shares are summed per output row in a fixed order.  A
// translation unit of its own, compiled beside the attention kernels.
#include <cuda_runtime.h>

#include "hq_decode_lane.cuh"
#include "hq_fused.h"
#include "hq_rows.cuh"

namespace hq {

// ---------------------------------------------------------------- weights
// x'[b][j] = s_dec * H * D * (R) x[b][j] for each 128-column tile j of
// activation row b (the whole matrix is one sign segment); 8 lanes a tile.
__global__ void __launch_bounds__(kRowThreads) rotate_x_kernel(GemmArgs a) {
  __shared__ __align__(16) float s_tr[(kRowThreads / 8) * kTrTile];
  const int tl = threadIdx.x >> 3, r = threadIdx.x & 7;
  const int64_t i = (int64_t)blockIdx.x * (kRowThreads / 8) + tl;   // (b, j)
  const bool valid = i < (int64_t)a.B * a.tpr;   // every lane stays for the transform
  const uint32_t mw = __ldg(a.dec.signs + (r >> 1)) >> (16 * (r & 1));
  rotate_row_t8(valid ? a.x + i * kTile : nullptr, (reinterpret_cast<uintptr_t>(a.x) & 15) == 0,
                a.dec.rot, mw, a.dec.s_dec, a.xrot + (valid ? i : 0) * kTile, s_tr + tl * kTrTile, r);
}

// Each tile's share of y.  A block decodes NG groups d apart, d = tpr /
// gcd(tpr, 32) -- their tiles fall on the same column blocks -- so each
// lane's slice of the rotated activations, read from L2 once, serves NG
// weight tiles (NG = 1 for a single activation row).  Lane r of tile t holds
// 16 lattice-domain values of each tile; partial dots with 8 activation rows
// at a time are reduced over the tile's 8 lanes by a butterfly that leaves
// one finished row on each lane.  When a weight row's tiles lie in one group
// (tpr divides 32, so d = 1) the block also sums each row's tile shares and
// writes y itself, in the order of gemm_reduce_kernel (one warp a row, lane
// l holding tile l, a fixed butterfly); otherwise the shares go to the
// workspace for that kernel.
template <int LAT, int K, int NG>
__global__ void __launch_bounds__(kDecThreads, NG > 2 ? 2 : 3) gemm_kernel(GemmArgs a, int pair_d) {
  __shared__ uint64_t s_start[kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[2][kDecThreads / 32];
  __shared__ float s_share[NG][8][kGroupTiles];  // (group, activation row of the chunk, tile)
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7;
  const int64_t bq = blockIdx.x / pair_d, bm = blockIdx.x - bq * pair_d;
  const int64_t g0 = NG * pair_d * bq + bm;      // groups g0 + n d, n < NG
  if (g0 >= a.dec.n_groups) return;              // uniform
  float e[NG][16];
  bool ok = true;
#pragma unroll
  for (int n = 0; n < NG; ++n) {
    const int64_t g = g0 + (int64_t)n * pair_d;
    if (g < a.dec.n_groups) {                    // uniform
      ok = decode_lane<LAT, K>(a.dec, g, e[n], s_start, s_warp) && ok;   // barriers inside
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) e[n][i] = 0.0f;
    }
  }
  if (!ok && tid == 0) atomicOr(a.dec.status, (uint32_t)HQ_ERR_CORRUPT);
  const int64_t tile0 = g0 * kGroupTiles + tl;
  const int64_t row = tile0 < a.dec.n_tiles ? div_by(tile0, a.tpr, a.tpr_shift) : 0;
  const int64_t j = tile0 < a.dec.n_tiles ? tile0 - row * a.tpr : 0;   // every tile's column block
  for (int b0 = 0; b0 < a.B; b0 += 8) {
    float p[NG][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float acc[NG];
#pragma unroll
      for (int n = 0; n < NG; ++n) acc[n] = 0.0f;
      if (b0 + i < a.B) {
        const float4 *xr = reinterpret_cast<const float4 *>(
            a.xrot + (int64_t)(b0 + i) * a.cols + j * kTile + 16 * r);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 xv = __ldg(xr + c);
#pragma unroll
          for (int n = 0; n < NG; ++n) {
            acc[n] = __fmaf_rn(xv.x, e[n][4 * c], acc[n]);
            acc[n] = __fmaf_rn(xv.y, e[n][4 * c + 1], acc[n]);
            acc[n] = __fmaf_rn(xv.z, e[n][4 * c + 2], acc[n]);
            acc[n] = __fmaf_rn(xv.w, e[n][4 * c + 3], acc[n]);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < NG; ++n) p[n][i] = acc[n];
    }
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
#pragma unroll
      for (int i = 0; i < m; ++i) {
        const bool upper = (r & m) != 0;
#pragma unroll
        for (int n = 0; n < NG; ++n) {
          const float send = upper ? p[n][i] : p[n][i + m], keep = upper ? p[n][i + m] : p[n][i];
          p[n][i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, m));
        }
      }
    }
    const int b = b0 + r;                        // slot kept by lane r is row b0 + r
    if (a.fold_rows) {                           // uniform: pair_d = 1, rows within groups
#pragma unroll
      for (int n = 0; n < NG; ++n) s_share[n][r][tl] = p[n][0];
      __syncthreads();
      const int lane = tid & 31, rpg = kGroupTiles / (int)a.tpr, nb = min(8, a.B - b0);
      const int per_n = 8 * rpg;
      for (int o = tid >> 5; o < NG * per_n; o += kDecThreads / 32) {   // (n, chunk row, weight row)
        const int n = o / per_n, bi = (o - n * per_n) / rpg, ol = o - n * per_n - bi * rpg;
        const int64_t g = g0 + n, orow = g * (kGroupTiles / a.tpr) + ol;
        if (bi >= nb || g >= a.dec.n_groups || orow >= a.rows) continue;   // warp-uniform
        float sum = lane < a.tpr ? __fadd_rn(0.0f, s_share[n][bi][ol * (int)a.tpr + lane]) : 0.0f;
#pragma unroll
        for (int dd = 16; dd >= 1; dd >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, dd));
        if (lane == 0) a.y[(int64_t)(b0 + bi) * a.rows + orow] = sum;
      }
      __syncthreads();                           // the next chunk rewrites the shares
    } else if (b < a.B) {
#pragma unroll
      for (int n = 0; n < NG; ++n) {
        const int64_t tile = tile0 + (int64_t)n * pair_d * kGroupTiles;
        if (g0 + (int64_t)n * pair_d < a.dec.n_groups && tile < a.dec.n_tiles)
          a.partial[(int64_t)b * a.dec.n_tiles + tile] = p[n][0];
      }
    }
  }
}

// y[b][o] = sum over the row's tiles of their shares: one warp per (b, o),
// lanes strided over the tiles, then a fixed butterfly (deterministic).
__global__ void gemm_reduce_kernel(GemmArgs a) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;   // (b, o)
  const int lane = threadIdx.x & 31;
  if (w >= (int64_t)a.B * a.rows) return;        // warp-uniform
  const int64_t b = w / a.rows, o = w - b * a.rows;
  const float *src = a.partial + b * a.dec.n_tiles + o * a.tpr;
  float s = 0.0f;
  for (int64_t jj = lane; jj < a.tpr; jj += 32) s = __fadd_rn(s, src[jj]);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, d));
  if (lane == 0) a.y[b * a.rows + o] = s;
}

constexpr int kGemmFourGroupRows = 16;  // from this many activation rows on, four groups a block

template <int LAT, int NG>
static void launch_gemm_k(const GemmArgs &a, int d, cudaStream_t st) {
  const int64_t blocks = (a.dec.n_groups + NG * d - 1) / (NG * d) * d;
  dim3 grid((unsigned)blocks), block(kDecThreads);
  // E8 (the weights' lattice) gets Rice k compiled in for the rates 3-5 bps;
  // the other lattices take k at run time (fewer instances to build)
  switch (LAT == 8 ? a.dec.rice_k : -1) {
    case 2: gemm_kernel<LAT, (LAT == 8 ? 2 : -1), NG><<<grid, block, 0, st>>>(a, d); break;
    case 3: gemm_kernel<LAT, (LAT == 8 ? 3 : -1), NG><<<grid, block, 0, st>>>(a, d); break;
    case 4: gemm_kernel<LAT, (LAT == 8 ? 4 : -1), NG><<<grid, block, 0, st>>>(a, d); break;
    default: gemm_kernel<LAT, -1, NG><<<grid, block, 0, st>>>(a, d); break;
  }
}

template <int LAT>
static void launch_gemm_lat(const GemmArgs &a, cudaStream_t st) {
  // groups d apart cover the same column blocks: 32 d is the first multiple
  // of tpr that is a multiple of 32
  int64_t g = 32, t = a.tpr;
  while (t != 0) {
    const int64_t m = g % t;
    g = t;
    t = m;
  }
  const int d = (int)(a.tpr / g);
  if (a.B < 2) launch_gemm_k<LAT, 1>(a, d, st);          // one activation row: decoding bounds it
  else if (a.B < kGemmFourGroupRows) launch_gemm_k<LAT, 2>(a, d, st);
  else launch_gemm_k<LAT, 4>(a, d, st);
}

int launch_decode_gemm(const GemmArgs &args, int lattice, cudaStream_t st) {
  GemmArgs a = args;
  a.fold_rows = kGroupTiles % a.tpr == 0 ? 1 : 0;
  const int64_t xt = (int64_t)a.B * a.tpr;
  rotate_x_kernel<<<(unsigned)((xt + kRowThreads / 8 - 1) / (kRowThreads / 8)), kRowThreads, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return 1;
  switch (lattice) {
    case 8: launch_gemm_lat<8>(a, st); break;
    case 4: launch_gemm_lat<4>(a, st); break;
    case 2: launch_gemm_lat<2>(a, st); break;
    default: launch_gemm_lat<1>(a, st); break;
  }
  if (cudaGetLastError() != cudaSuccess) return 1;
  if (a.fold_rows) return 0;                     // y written by the product kernel
  const int64_t warps = (int64_t)a.B * a.rows;
  gemm_reduce_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace hq

// hq_fused.cu -- kernels that consume compressed tiles without writing them
// out: attention scores from compressed K (hq_decode_qk) and decode attention
// over compressed K and V (hq_decode_attention) -- the summary's closing
// section, fused decode + MMA (the products with compressed weights are in
// hq_fused_gemm.cu).  Each decodes only to the lattice domain e = v - u with
// the shared decoding step and moves the transform to the other operand:
// queries are rotated once into that domain (q' = s_dec H D R q), and the
// attention output rows are transformed back once per row.
#include <cuda_runtime.h>

#include <cmath>

#include "hq_decode_lane.cuh"
#include "hq_fused.h"
#include "hq_rows.cuh"
#include "hq_umma.cuh"

namespace hq {

// q'[row] = s_dec * H * D_h * (R_h) q[row] for row = b * Hq + hq,
// h = hq / (Hq / n_kv), R_h the optional dense rotation of h's segment; 8
// lanes a row.
__global__ void __launch_bounds__(kRowThreads) rotate_queries_kernel(QkArgs a) {
  __shared__ __align__(16) float s_tr[(kRowThreads / 8) * kTrTile];
  const int tl = threadIdx.x >> 3, r = threadIdx.x & 7;
  const int row = blockIdx.x * (kRowThreads / 8) + tl;
  const bool valid = row < a.B * a.Hq;           // every lane stays for the transform
  const int hq = (valid ? row : 0) % a.Hq, h = hq / (a.Hq / a.n_kv);
  const int64_t seg = div_by((int64_t)h * a.n_tokens, a.dec.tiles_per_segment, a.dec.seg_shift);
  const uint32_t mw = __ldg(a.dec.signs + 4 * seg + (r >> 1)) >> (16 * (r & 1));
  rotate_row_t8(valid ? a.q + (int64_t)row * kTile : nullptr,
                (reinterpret_cast<uintptr_t>(a.q) & 15) == 0,
                a.dec.rot != nullptr ? a.dec.rot + seg * (int64_t)(kTile * kTile) : nullptr, mw,
                a.dec.s_dec, a.qrot + (int64_t)(valid ? row : 0) * kTile, s_tr + tl * kTrTile, r);
}

// Scores of one KV head over a chunk of its token groups for one tile of
// up to 64 query rows, on the tensor cores (tcgen05, kind::f16 with fp16
// operands, fp32 accumulator in tensor memory).  Each query row and each
// token's e is scaled by a power of two to below 1 in magnitude, then split
// into two fp16 parts, x = x_1 + x_2 (|x - x_1 - x_2| <= 2^-22 |x| + 2^-25),
// and the fp32-level product is laid along K: A = [q_1 | q_1 | q_2] and
// B = [e_1 | e_2 | e_1] over K = 3 x 128, so one accumulator lane per query
// row receives q_1 e_1 + q_1 e_2 + q_2 e_1 (the dropped q_2 e_2 is below
// 2^-22 of the product); the epilogue multiplies by the two inverse scales
// (exact).  M = 128 with rows 64..127 of A aliasing the next K-core (their
// results are never read), N = 32 tokens of a group.
//
// The block holds the split query rows once and runs four independent teams
// of 256 threads (named barriers), each decoding every fourth group of the
// chunk into its own B and accumulator columns: a team decodes its next group
// while the MMAs of its previous one run, then writes that group's scores
// from tensor memory.  With 16-bit operands (99 KB) and 32 registers per
// thread two blocks fit on an SM, 64 warps of decoding.  Dimensions are
// permuted consistently in A and B (16-byte block 2 r + c of d, dimensions
// 16 r + 8 c .. +7, goes to K-core 8 c + r) so that the eight lanes of a
// tile store e to distinct banks.
constexpr int kQkRows = 64;                      // query rows per block
constexpr int kQkTeams = 4;
constexpr int kQkThreads = kQkTeams * kDecThreads;
constexpr int kQkBlocksPerSm = 2;
constexpr int kQkChunkMin = kQkTeams, kQkChunkMax = 32;   // groups of 32 tokens per block
constexpr int kQkCores = kTile / 8;              // K-cores of one fp16 part (8 dimensions each)
constexpr int kQkAKStride = 1024;                // bytes between K-cores of A (8 row groups)
constexpr int kQkAGStride = 128;                 // bytes between 8-row groups of A
constexpr int kQkBKStride = 528;                 // bytes between K-cores of B (4 token groups + 16)
constexpr int kQkBGStride = 128;                 // bytes between 8-token groups of B
constexpr int kQkABytes = 2 * kQkCores * kQkAKStride + 1024;   // [q_1 | q_2] + the aliased rows' reach
constexpr int kQkBBytes = 2 * kQkCores * kQkBKStride;          // [e_1 | e_2] of one team
constexpr int kQkSmemBytes = kQkABytes + kQkTeams * kQkBBytes;
constexpr uint32_t kQkIdesc = umma_idesc_f16(128, 32);
constexpr uint32_t kQkTmemCols = 32 * kQkTeams;
static_assert(kQkRows * kQkCores == kQkThreads, "one (row, 8-dimension block) of A per thread");

__device__ __forceinline__ void st_shared16(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// The lane's 16 values of e (one token, dimensions 16 r .. 16 r + 15), scaled
// by `sc` and split into fp16 parts: block c (dimensions 16 r + 8 c .. +7) of
// e_1 at K-core 8 c + r (`dst` = K-core r of the token's row), e_2 a part
// further on.
__device__ __forceinline__ void qk_store_b(uint32_t dst, const float e[16], float sc) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      upk2(mul2(pk2(e[8 * c + 2 * i], e[8 * c + 2 * i + 1]), pk2(sc, sc)), x[2 * i], x[2 * i + 1]);
    uint4 hi, lo;
    split_f16x2(x[0], x[1], hi.x, lo.x);
    split_f16x2(x[2], x[3], hi.y, lo.y);
    split_f16x2(x[4], x[5], hi.z, lo.z);
    split_f16x2(x[6], x[7], hi.w, lo.w);
    st_shared16(dst + 8 * c * kQkBKStride, hi);
    st_shared16(dst + (8 * c + kQkCores) * kQkBKStride, lo);
  }
}

// A token's e into B: the largest |e| over the token's 8 lanes sets its
// power-of-two scale; lane 0 of the tile keeps the inverse for the epilogue.
// All 32 lanes of the warp must call it.
__device__ __forceinline__ void qk_put_e(const float e[16], uint32_t dst, float *tinv, int tl, int r) {
  float m = fabsf(e[0]);
#pragma unroll
  for (int i = 1; i < 16; ++i) m = fmaxf(m, fabsf(e[i]));
#pragma unroll
  for (int d = 1; d < 8; d <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if (r == 0) tinv[tl] = inv_scale_of(m);
  qk_store_b(dst, e, scale_of(m));
}

template <int LAT, int K>
__global__ void __launch_bounds__(kQkThreads, kQkBlocksPerSm) scores_kernel(QkArgs a, int chunk_groups) {
  __shared__ uint64_t s_start[kQkTeams][kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[kQkTeams][2][kDecThreads / 32];
  __shared__ __align__(8) uint64_t s_bar[kQkTeams];
  __shared__ uint32_t s_taddr;
  __shared__ uint32_t s_qmax[kQkRows];           // largest |q'| of each row (float bits)
  __shared__ __align__(16) float s_tinv[kQkTeams][2][kGroupTiles];   // 1 / token scale, two groups
  extern __shared__ __align__(128) unsigned char s_ops[];   // A | B of team 0 | ... | B of team 3
  const int team = threadIdx.x / kDecThreads, tid = TeamBar::tid();
  const int tl = tid >> 3, r = tid & 7, warp = tid >> 5;
  const int chunk = blockIdx.x, h = blockIdx.y, row0 = blockIdx.z * kQkRows;
  const int64_t T = a.n_tokens;
  const int G = a.Hq / a.n_kv, rows = a.B * G;
  const int64_t tile_lo = (int64_t)h * T, tile_hi = tile_lo + T;
  const int64_t g_first = tile_lo / kGroupTiles, g_end = (tile_hi - 1) / kGroupTiles + 1;
  const int64_t gb = g_first + (int64_t)chunk * chunk_groups;
  const int64_t ge = min(gb + (int64_t)chunk_groups, g_end);
  if (gb >= ge) return;                          // uniform: nothing of head h here
  if (threadIdx.x < 32) tmem_alloc(&s_taddr, kQkTmemCols);
  if (tid == 32) mbar_init(&s_bar[team], 1);
  if (threadIdx.x < kQkRows) s_qmax[threadIdx.x] = 0u;
  // A: the block's rotated query rows, each scaled by a power of two to below
  // 1 and split into fp16 parts (rows past the end are zeros); thread =
  // (8-dimension block db, row q), 8 rows per 128-byte phase
  {
    const int q = threadIdx.x & (kQkRows - 1), db = threadIdx.x >> 6, row = row0 + q;
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
    if (row < rows) {
      const int b = row / G, gq = row - b * G;
      const float4 *src = reinterpret_cast<const float4 *>(
                              a.qrot + ((int64_t)b * a.Hq + (int64_t)h * G + gq) * kTile) + 2 * db;
      v0 = __ldg(src);
      v1 = __ldg(src + 1);
    }
    const float m = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                          fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
    __syncthreads();                             // s_qmax cleared
    atomicMax(&s_qmax[q], __float_as_uint(m));   // nonnegative floats order as integers
    __syncthreads();
    const float sc = scale_of(__uint_as_float(s_qmax[q]));
    uint4 hi, lo;
    split_f16x2(__fmul_rn(v0.x, sc), __fmul_rn(v0.y, sc), hi.x, lo.x);
    split_f16x2(__fmul_rn(v0.z, sc), __fmul_rn(v0.w, sc), hi.y, lo.y);
    split_f16x2(__fmul_rn(v1.x, sc), __fmul_rn(v1.y, sc), hi.z, lo.z);
    split_f16x2(__fmul_rn(v1.z, sc), __fmul_rn(v1.w, sc), hi.w, lo.w);
    const int core = 8 * (db & 1) + (db >> 1);
    unsigned char *dst = s_ops + (q >> 3) * kQkAGStride + core * kQkAKStride + (q & 7) * 16;
    *reinterpret_cast<uint4 *>(dst) = hi;
    *reinterpret_cast<uint4 *>(dst + kQkCores * kQkAKStride) = lo;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t dcol = s_taddr + (uint32_t)(32 * team);
  const uint32_t a_op = smem_addr(s_ops), b_op = a_op + kQkABytes + team * kQkBBytes;
  const uint32_t bdst = b_op + (tl >> 3) * kQkBGStride + (tl & 7) * 16 + r * kQkBKStride;
  uint64_t *const bar = &s_bar[team];
  // epilogue geometry: team warps 0, 1, 4, 5 read lanes (query rows)
  // 32 (w % 4) + lane, tokens 16 (w / 4) .. +15 of the group
  const bool reader = (warp & 2) == 0;
  const int q_row = 32 * (warp & 1) + (tid & 31), row = row0 + q_row, tcol = 16 * (warp >> 2);
  const float qinv = inv_scale_of(__uint_as_float(s_qmax[q_row]));
  float *srow = nullptr;
  if (reader && row < rows) {
    const int b = row / G, gq = row - b * G;
    srow = a.scores + ((int64_t)b * a.Hq + (int64_t)h * G + gq) * T - tile_lo;
  }
  bool ok_wait = true;                           // team-uniform after each barrier
  int committed = 0;
  // this team's groups gb + team, gb + team + 4, ...; the step past the last
  // one only drains
  for (int64_t g = gb + team; g < ge + kQkTeams; g += kQkTeams) {
    const bool has = g < ge;
    float e[16];
    bool lane_ok = true;                         // this lane's decoding verdict
    if (has) lane_ok = decode_lane<LAT, K, TeamBar, true>(a.dec, g, e, s_start[team], s_warp[team]);
    if (committed > 0 && ok_wait) {              // the previous group: wait, then its scores
      // warp-uniform for the tensor-memory loads; team-uniform at the next barrier
      ok_wait = __all_sync(0xffffffffu, mbar_wait(bar, (uint32_t)(committed - 1) & 1u, 1u << 22));
      if (ok_wait && has) qk_put_e(e, bdst, s_tinv[team][committed & 1], tl, r);   // B is free again
      if (ok_wait && reader) {                   // two loads of 8 columns (32 registers)
        tc_fence_after();
        const float *tinv = s_tinv[team][(committed - 1) & 1] + tcol;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[8];
          tmem_ld8(dcol + ((uint32_t)(32 * (warp & 1)) << 16) + (uint32_t)(tcol + 8 * hh), v);
          const float4 i0 = *reinterpret_cast<const float4 *>(tinv + 8 * hh);
          const float4 i1 = *reinterpret_cast<const float4 *>(tinv + 8 * hh + 4);
          const float ti[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(__fmul_rn(v[j], qinv), ti[j]);
          const int64_t t0 = (g - kQkTeams) * kGroupTiles + tcol + 8 * hh;
          if (srow != nullptr) {
            if (t0 >= tile_lo && t0 + 8 <= tile_hi) {
              float4 *dst = reinterpret_cast<float4 *>(srow + t0);
              if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                dst[1] = make_float4(v[4], v[5], v[6], v[7]);
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) srow[t0 + j] = v[j];
              }
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (t0 + j >= tile_lo && t0 + j < tile_hi) srow[t0 + j] = v[j];
            }
          }
        }
      }
    } else if (has) {                            // first group of the team (or after a timeout)
      qk_put_e(e, bdst, s_tinv[team][committed & 1], tl, r);
    }
    if (!has) continue;
    fence_async_smem();
    tc_fence_before();
    // one barrier for the group's decoding verdicts and the previous wait;
    // only when something failed, two more sort out which (rare)
    if (TeamBar::sync_or(!(lane_ok && ok_wait)) != 0) {
      const bool corrupt = TeamBar::sync_or(!lane_ok) != 0;
      ok_wait = TeamBar::sync_and(ok_wait) != 0;
      if (corrupt) {                             // the group decodes to zeros
        if (tid == 0) atomicOr(a.dec.status, (uint32_t)HQ_ERR_CORRUPT);
        const float zeros[16] = {};
        qk_store_b(bdst, zeros, 1.0f);
        fence_async_smem();
        TeamBar::sync();
      }
    }
    if (!ok_wait) continue;
    ++committed;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const int ka = part == 2 ? kQkCores : 0, kb = part == 1 ? kQkCores : 0;
#pragma unroll
        for (int ks = 0; ks < kQkCores / 2; ++ks)
          umma_f16(dcol, umma_desc(a_op + (ka + 2 * ks) * kQkAKStride, kQkAKStride, kQkAGStride),
                    umma_desc(b_op + (kb + 2 * ks) * kQkBKStride, kQkBKStride, kQkBGStride), kQkIdesc,
                    (part > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(bar);
    }
  }
  if (!ok_wait) {
    if (tid == 0) atomicOr(a.dec.status, (uint32_t)HQ_ERR_TIMEOUT);
    if (committed > 0) mbar_wait(bar, (uint32_t)(committed - 1) & 1u, 1u << 22);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(s_taddr, kQkTmemCols);
  }
}

// ---------------------------------------------------------------- attention
// Softmax over the tokens of one query row, in place (only when the caller
// asks for the probabilities): p = exp(z - m) / l with
// z = fl(scale * s), m = max z and l = sum of exp(z - m) (per-thread running
// maximum and rescaled sum, then combined over the block).
constexpr int kSoftmaxThreads = 256;
__device__ __forceinline__ void ml_combine(float &m, float &l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  const float a = (m == M) ? l : __fmul_rn(l, expf(__fsub_rn(m, M)));
  const float b = (m2 == M) ? l2 : __fmul_rn(l2, expf(__fsub_rn(m2, M)));
  m = M;
  l = __fadd_rn(a, b);
}

__global__ void __launch_bounds__(kSoftmaxThreads) softmax_kernel(AttnArgs a) {
  __shared__ float s_m[kSoftmaxThreads / 32], s_l[kSoftmaxThreads / 32];
  const int64_t T = a.qk.n_tokens;
  float *row = a.qk.scores + (int64_t)blockIdx.x * T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m = -INFINITY, l = 0.0f;
  for (int64_t t = tid; t < T; t += kSoftmaxThreads) {
    const float z = __fmul_rn(row[t], a.scale);
    if (z > m) {
      l = __fmul_rn(l, expf(__fsub_rn(m, z)));   // l is 0 while m is -inf
      m = z;
    }
    l = __fadd_rn(l, expf(__fsub_rn(z, m)));
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, d), l2 = __shfl_xor_sync(0xffffffffu, l, d);
    ml_combine(m, l, m2, l2);
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
  __syncthreads();
  m = s_m[0];
  l = s_l[0];
#pragma unroll
  for (int w = 1; w < kSoftmaxThreads / 32; ++w) ml_combine(m, l, s_m[w], s_l[w]);
  for (int64_t t = tid; t < T; t += kSoftmaxThreads) {
    const float z = __fmul_rn(row[t], a.scale);
    row[t] = __fdiv_rn(expf(__fsub_rn(z, m)), l);
  }
}

// Partial sums of one KV head over a chunk of its token groups, in the
// lattice domain and in flash-decoding form: the block reduces the chunk's
// scaled scores z to m = max z and l = sum exp(z - m) per query row, then
// accumulates sum_t exp(z_t - m) e_t with V's tiles decoded only to
// e = v - u (no inverse transform per token), since
// sum_t p_t Vhat_t = D s_dec H (sum_t p_t e_t) up to rounding;
// pv_finish_kernel combines the chunks and applies H, s_dec and D once per
// query row.  Tokens of the group outside head h (a group that straddles two
// heads) get weight 0.
//
// The contraction runs on the tensor cores (tcgen05, kind::tf32, fp32
// accumulator in tensor memory): per group, D[d][n] += sum_t E^T[d][t] B[n][t]
// with M = 128 dimensions d, K = 32 tokens and N = 128 columns that stack the
// tf32 split of the weights, B = [p_hi (64 rows); p_lo (64 rows)], each issued
// twice (A = e_hi^T, then e_lo^T).  The four partial products of the split
// operands give an fp32-level result: column n of D holds (e_hi + e_lo) p_hi
// and column 64 + n holds (e_hi + e_lo) p_lo of row n.
//
// A block runs four independent teams of 256 threads (named barriers), each
// decoding every fourth group of the chunk into operands and an accumulator
// of its own, and decoding its next group while the MMAs of the previous one
// run; at the end the teams' sums are added in team order (deterministic).
// Operand layout: K-cores 2064 bytes apart (eight 8-row groups of 128 bytes
// plus 16), so that consecutive K-cores fall on rotated banks without
// padding; the rows of e^T are permuted (dimension 16 r + c of lane r goes to
// row 8 (2 r + c / 8) + (c + r) % 8) so that the eight lanes of a tile store
// to distinct banks.  The permutation is undone when the sums are read.
constexpr int kPvTeams = 4;
constexpr int kPvThreads = kPvTeams * kDecThreads;
constexpr int kPvKStride = 2064;                 // bytes between K-cores
constexpr int kPvGStride = 128;                  // bytes between 8-row groups
constexpr int kPvOpBytes = 7 * kPvKStride + 16 * kPvGStride;   // 16496 per operand
constexpr int kPvTeamBytes = 3 * kPvOpBytes;     // e_hi^T | e_lo^T | B
constexpr int kPvSmemBytes = kPvTeams * kPvTeamBytes;
static_assert(kPvTeams * kPvRows * kTile * 4 <= kPvSmemBytes, "team sums fit the operand area");
constexpr uint32_t kPvIdesc = umma_idesc_tf32(128, 128);
constexpr uint32_t kPvTmemCols = 128 * kPvTeams;
constexpr uint32_t kPvWaitLimit = 1u << 22;
constexpr int kPvChunkMax = 32;                  // largest chunk the launch may pick (groups)

// This thread's 8 scaled scores z = fl(scale s) of group g (element
// i = tid + 256 k of the group's 64 rows x 32 tokens, row-major, tid the
// thread's index in its team): consecutive threads read consecutive tokens
// of one row; tokens outside head h or rows past the end read as -inf
// (probability 0).
__device__ __forceinline__ void pv_load_z(const AttnArgs &a, int64_t g, int h, int row0, int G,
                                          int rows, int64_t tile_lo, int64_t tile_hi, int tid,
                                          float z[8]) {
  const int64_t T = a.qk.n_tokens;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = tid + k * kDecThreads;
    const int rr = i >> 5, j = i & 31;
    const int64_t tile = g * kGroupTiles + j;
    const int row = row0 + rr;
    z[k] = -INFINITY;
    if (tile >= tile_lo && tile < tile_hi && row < rows) {
      const int b = row / G, gq = row - b * G;
      z[k] = __fmul_rn(a.qk.scores[((int64_t)b * a.qk.Hq + (int64_t)h * G + gq) * T +
                                   (tile - tile_lo)], a.scale);
    }
  }
}
template <int LAT, int K>
__global__ void __launch_bounds__(kPvThreads, 1) pv_kernel(AttnArgs a) {
  __shared__ uint64_t s_start[kPvTeams][kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[kPvTeams][2][kDecThreads / 32];
  __shared__ float s_m[kPvRows];
  __shared__ float s_l[kPvTeams][kPvRows];
  __shared__ __align__(8) uint64_t s_bar[kPvTeams];
  __shared__ uint32_t s_taddr;
  extern __shared__ __align__(128) unsigned char s_ops[];   // team 0 | ... | team 3
  const int team = threadIdx.x / kDecThreads, tid = TeamBar::tid();
  const int tl = tid >> 3, r = tid & 7, warp = tid >> 5, lane = tid & 31;
  const int chunk = blockIdx.x, h = blockIdx.y, rt = blockIdx.z;
  const int64_t T = a.qk.n_tokens;
  const int Hq = a.qk.Hq, G = Hq / a.qk.n_kv, rows = a.qk.B * G, row0 = rt * kPvRows;
  const int64_t tile_lo = (int64_t)h * T, tile_hi = tile_lo + T;
  const int64_t g_first = tile_lo / kGroupTiles, g_end = (tile_hi - 1) / kGroupTiles + 1;
  const int64_t gb = g_first + (int64_t)chunk * a.pv_chunk;
  const int64_t ge = min(gb + (int64_t)a.pv_chunk, g_end);
  if (threadIdx.x < 32) tmem_alloc(&s_taddr, kPvTmemCols);
  if (tid == 32) mbar_init(&s_bar[team], 1);
  // this chunk's softmax maximum per row, m = max z over its tokens: block
  // warp w takes rows w and w + 32, its lanes consecutive tokens, 256 at a
  // time; l = sum exp(z - m) is summed from the weights of the main loop
  // below
  {
    const int64_t c_lo = max(gb * kGroupTiles, tile_lo), c_hi = min(ge * kGroupTiles, tile_hi);
    for (int rr = threadIdx.x >> 5; rr < kPvRows; rr += kPvThreads / 32) {
      const int row = row0 + rr;
      float m = -INFINITY;
      if (row < rows) {
        const int b = row / G, gq = row - b * G;
        const float *srow = a.qk.scores + ((int64_t)b * Hq + (int64_t)h * G + gq) * T - tile_lo;
        for (int64_t t0 = c_lo; t0 < c_hi; t0 += 256) {
          float z[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int64_t t = t0 + lane + 32 * j;
            z[j] = t < c_hi ? __fmul_rn(srow[t], a.scale) : -INFINITY;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) m = fmaxf(m, z[j]);
        }
      }
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
      if (lane == 0) s_m[rr] = m;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t dcol = s_taddr + (uint32_t)(128 * team);
  unsigned char *const tops = s_ops + team * kPvTeamBytes;
  const uint32_t a_hi = smem_addr(tops), a_lo = a_hi + kPvOpBytes, b_op = a_hi + 2 * kPvOpBytes;
  // e^T slots of this lane (token tl, rows of dimensions 16 r .. 16 r + 15)
  unsigned char *const ebase = tops + 256 * r + (tl >> 2) * kPvKStride + (tl & 3) * 4;
  // B slots: rows (tid >> 5) + 8 k (p_hi) and 64 + (tid >> 5) + 8 k (p_lo), token lane
  float *const bp = reinterpret_cast<float *>(tops + 2 * kPvOpBytes + 16 * warp +
                                              (lane >> 2) * kPvKStride + (lane & 3) * 4);
  uint64_t *const bar = &s_bar[team];
  bool ok_wait = true;                           // team-uniform after each barrier
  int committed = 0;                             // groups whose MMAs were issued
  float pn[8], lsum[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) lsum[k] = 0.0f;
  for (int64_t g = gb + team; g < ge; g += kPvTeams) {   // team-uniform bounds
    float e[16];
    const bool lane_ok = decode_lane<LAT, K, TeamBar, true>(a.v, g, e, s_start[team], s_warp[team]);
    pv_load_z(a, g, h, row0, G, rows, tile_lo, tile_hi, tid, pn);
    // the MMAs of the team's previous group must be done with the operands
    if (committed > 0 && ok_wait) ok_wait = mbar_wait(bar, (uint32_t)(committed - 1) & 1u, kPvWaitLimit);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float hi, lo;
      split_tf32(e[c], hi, lo);
      const int off = 128 * (c >> 3) + ((16 * r + 16 * c) & 0x70);   // permuted row
      *reinterpret_cast<float *>(ebase + off) = hi;
      *reinterpret_cast<float *>(ebase + kPvOpBytes + off) = lo;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {                // p = exp(z - m), 0 for z = -inf
      const float mm = s_m[warp + 8 * k];
      const float p = pn[k] == -INFINITY ? 0.0f : expf(__fsub_rn(pn[k], mm));
      lsum[k] = __fadd_rn(lsum[k], p);           // this lane's token column, in group order
      float hi, lo;
      split_tf32(p, hi, lo);
      bp[k * kPvGStride / 4] = hi;
      bp[(k + 8) * kPvGStride / 4] = lo;
    }
    fence_async_smem();
    // one barrier for the group's decoding verdicts and the previous wait;
    // only when something failed, two more sort out which (rare)
    if (TeamBar::sync_or(!(lane_ok && ok_wait)) != 0) {
      const bool corrupt = TeamBar::sync_or(!lane_ok) != 0;
      ok_wait = TeamBar::sync_and(ok_wait) != 0;
      if (corrupt) {                             // the group's values decode to zeros
        if (tid == 0) atomicOr(a.v.status, (uint32_t)HQ_ERR_CORRUPT);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int off = 128 * (c >> 3) + ((16 * r + 16 * c) & 0x70);
          *reinterpret_cast<float *>(ebase + off) = 0.0f;
          *reinterpret_cast<float *>(ebase + kPvOpBytes + off) = 0.0f;
        }
        fence_async_smem();
        TeamBar::sync();
      }
    }
    if (!ok_wait) continue;
    const bool first = committed == 0;
    ++committed;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_tf32(dcol, umma_desc(a_hi + ks * 2 * kPvKStride, kPvKStride, kPvGStride),
                  umma_desc(b_op + ks * 2 * kPvKStride, kPvKStride, kPvGStride), kPvIdesc,
                  (!first || ks > 0) ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_tf32(dcol, umma_desc(a_lo + ks * 2 * kPvKStride, kPvKStride, kPvGStride),
                  umma_desc(b_op + ks * 2 * kPvKStride, kPvKStride, kPvGStride), kPvIdesc, 1u);
      umma_commit(bar);
    }
  }
  // the team's l per row: its lanes' column sums combined by a fixed butterfly
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float l = lsum[k];
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, d));
    if (lane == 0) s_l[team][warp + 8 * k] = l;
  }
  if (committed > 0 && ok_wait)                  // the team's last MMAs
    ok_wait = mbar_wait(bar, (uint32_t)(committed - 1) & 1u, kPvWaitLimit);
  ok_wait = __all_sync(0xffffffffu, ok_wait) != 0;   // warp-uniform for the tensor-memory loads
  tc_fence_before();
  __syncthreads();                               // every team's operands are free
  tc_fence_after();
  // the team's sums, hi + lo halves added, as S[team][row][d] in the operand
  // area: warp w reads tensor-memory lanes (permuted rows of e^T)
  // 32 (w % 4) .. +31 for query rows 32 (w / 4) .. +31
  {
    float *S = reinterpret_cast<float *>(s_ops) + team * (kPvRows * kTile);
    const int L = 32 * (warp & 3) + lane, Gr = L >> 3, rr = Gr >> 1;
    const int d = 16 * rr + 8 * (Gr & 1) + (((L & 7) - rr) & 7);
    const int hf = warp >> 2;
    if (committed > 0 && ok_wait) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float vh[16], vl[16];
        const uint32_t lane_addr = dcol + ((uint32_t)(32 * (warp & 3)) << 16);
        tmem_ld16(lane_addr + (uint32_t)(32 * hf + 16 * jj), vh);
        tmem_ld16(lane_addr + (uint32_t)(64 + 32 * hf + 16 * jj), vl);
#pragma unroll
        for (int j = 0; j < 16; ++j) S[(32 * hf + 16 * jj + j) * kTile + d] = __fadd_rn(vh[j], vl[j]);
      }
    } else {                                     // no group of this team (or a lost wait)
#pragma unroll
      for (int j = 0; j < 32; ++j) S[(32 * hf + j) * kTile + d] = 0.0f;
    }
  }
  if (!ok_wait) {
    atomicOr(a.v.status, (uint32_t)HQ_ERR_TIMEOUT);
    // the team's last MMAs may still be in flight: give them a bounded
    // while before the tensor memory goes back
    if (committed > 0) mbar_wait(bar, (uint32_t)(committed - 1) & 1u, kPvWaitLimit);
  }
  tc_fence_before();
  __syncthreads();
  // partial sums and statistics of the block: teams added in order
  {
    const float *S = reinterpret_cast<const float *>(s_ops);
    float *part = a.partials + ((((int64_t)h * a.chunks + chunk) * a.rowtiles + rt) * kPvRows) * kTile;
    for (int i = threadIdx.x; i < kPvRows * kTile; i += kPvThreads) {
      float v = S[i];
#pragma unroll
      for (int t = 1; t < kPvTeams; ++t) v = __fadd_rn(v, S[t * kPvRows * kTile + i]);
      part[i] = v;
    }
    if (threadIdx.x < kPvRows) {
      const int rr = threadIdx.x;
      float l = s_l[0][rr];
#pragma unroll
      for (int t = 1; t < kPvTeams; ++t) l = __fadd_rn(l, s_l[t][rr]);
      a.stats[(((int64_t)h * a.chunks + chunk) * a.rowtiles + rt) * kPvRows + rr] = make_float2(s_m[rr], l);
    }
  }
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(s_taddr, kPvTmemCols);
  }
}

// out[b][hq] = D_h * fl(H (sum_c w_c acc_c / sum_c w_c l_c) * s_dec) with
// w_c = exp(m_c - max_c m_c): the chunks' softmax pieces rescaled to a common
// maximum and summed in chunk order; one block of 128 threads per query row.
__global__ void __launch_bounds__(kTile) pv_finish_kernel(AttnArgs a) {
  __shared__ float x[kTile];
  const int row = blockIdx.x, d = threadIdx.x;
  const int Hq = a.qk.Hq, G = Hq / a.qk.n_kv;
  const int b = row / Hq, hq = row - b * Hq, h = hq / G;
  const int rr = b * G + (hq - h * G), rt = rr / kPvRows, rl = rr - rt * kPvRows;
  const float2 *st = a.stats + ((int64_t)h * a.chunks * a.rowtiles + rt) * kPvRows + rl;
  const int64_t cstride = (int64_t)a.rowtiles * kPvRows;
  float M = -INFINITY;
  for (int c = 0; c < a.chunks; ++c) M = fmaxf(M, st[c * cstride].x);
  float L = 0.0f, s = 0.0f;
  for (int c = 0; c < a.chunks; ++c) {
    const float2 ml = st[c * cstride];
    if (ml.x == -INFINITY) continue;             // a chunk without tokens of this head
    const float w = expf(__fsub_rn(ml.x, M));
    L = __fadd_rn(L, __fmul_rn(w, ml.y));
    s = __fadd_rn(s, __fmul_rn(w, a.partials[((((int64_t)h * a.chunks + c) * a.rowtiles + rt) *
                                                  kPvRows + rl) * kTile + d]));
  }
  x[d] = __fdiv_rn(s, L);
  __syncthreads();
#pragma unroll
  for (int hh = 1; hh < kTile; hh <<= 1) {
    const float mine = x[d], other = x[d ^ hh];
    __syncthreads();
    x[d] = (d & hh) ? __fsub_rn(other, mine) : __fadd_rn(mine, other);
    __syncthreads();
  }
  const int64_t seg = div_by((int64_t)h * a.qk.n_tokens, a.v.tiles_per_segment, a.v.seg_shift);
  const uint32_t mw = __ldg(a.v.signs + 4 * seg + (d >> 5));
  const float y = __fmul_rn(x[d], a.v.s_dec);
  const float yd = ((mw >> (d & 31)) & 1u) ? -y : y;
  if (a.v.rot == nullptr) {
    a.out[(int64_t)row * kTile + d] = yd;
    return;
  }
  // dense rotation of the values: out = R^T y, one chain over i per output
  const float *R = a.v.rot + seg * (int64_t)(kTile * kTile);
  __syncthreads();
  x[d] = yd;
  __syncthreads();
  float acc = 0.0f;
  for (int i = 0; i < kTile; ++i) acc = __fmaf_rn(__ldg(R + i * kTile + d), x[i], acc);
  a.out[(int64_t)row * kTile + d] = acc;
}

// The chunk size in [lo, hi] groups whose grid (chunks x `other` blocks)
// fills the most of its last wave of `cap` resident blocks; ties go to the
// larger chunk.  Chunks above max_chunks (when positive) are not allowed.
static int pick_chunk(int64_t groups, int64_t other, int cap, int lo, int hi, int64_t max_chunks) {
  double best = -1.0;
  int pick = lo;
  for (int cs = hi; cs >= lo; --cs) {
    const int64_t chunks = (groups + cs - 1) / cs;
    if (max_chunks > 0 && chunks > max_chunks) continue;
    const double waves = (double)(chunks * other) / cap, fill = waves / std::ceil(waves);
    if (fill > best + 1e-9) {
      best = fill;
      pick = cs;
    }
  }
  return pick;
}

// Resident blocks of a kernel instance per SM, times the SM count of the
// current device (kept per call site and device after the first query).
template <class F>
static int capacity(int *cache, F kernel, int threads, int smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0, per_sm = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  const int c = sms * per_sm > 0 ? sms * per_sm : 1;
  if (dev >= 0 && dev < 64) cache[dev] = c;
  return c;
}

template <int LAT, int K>
static void launch_qk_one(const QkArgs &a, cudaStream_t st) {
  static int cache[64] = {};
  const int cap = capacity(cache, scores_kernel<LAT, K>, kQkThreads, kQkSmemBytes);
  // a head's tokens touch at most ceil(T / 32) + 1 groups
  const int64_t groups = (a.n_tokens + kGroupTiles - 1) / kGroupTiles + 1;
  const int rowtiles = (a.B * (a.Hq / a.n_kv) + kQkRows - 1) / kQkRows;
  const int cs = pick_chunk(groups, (int64_t)a.n_kv * rowtiles, cap, kQkChunkMin, kQkChunkMax, 0);
  dim3 grid((unsigned)((groups + cs - 1) / cs), (unsigned)a.n_kv, (unsigned)rowtiles),
      block(kQkThreads);
  scores_kernel<LAT, K><<<grid, block, kQkSmemBytes, st>>>(a, cs);
}

template <int LAT>
static void launch_qk_lat(const QkArgs &a, cudaStream_t st) {
  switch (a.dec.rice_k) {
    case 1: launch_qk_one<LAT, 1>(a, st); break;
    case 2: launch_qk_one<LAT, 2>(a, st); break;
    case 3: launch_qk_one<LAT, 3>(a, st); break;
    default: launch_qk_one<LAT, -1>(a, st); break;
  }
}

// The chunk size is picked for whole waves (pick_chunk); the workspace holds
// the chunks of the smallest chunk size, a.chunks on entry.
template <int LAT, int K>
static void launch_pv_k(AttnArgs a, cudaStream_t st) {
  static int cache[64] = {};
  const int cap = capacity(cache, pv_kernel<LAT, K>, kPvThreads, kPvSmemBytes);
  const int64_t groups = (a.qk.n_tokens + kGroupTiles - 1) / kGroupTiles + 1;   // a head's, at most
  a.pv_chunk = pick_chunk(groups, (int64_t)a.qk.n_kv * a.rowtiles, cap, kPvMinGroupsPerChunk,
                          kPvChunkMax, a.chunks);
  a.chunks = (int)((groups + a.pv_chunk - 1) / a.pv_chunk);
  dim3 grid((unsigned)a.chunks, (unsigned)a.qk.n_kv, (unsigned)a.rowtiles), block(kPvThreads);
  pv_kernel<LAT, K><<<grid, block, kPvSmemBytes, st>>>(a);
  pv_finish_kernel<<<(unsigned)(a.qk.B * a.qk.Hq), kTile, 0, st>>>(a);
}

template <int LAT>
static void launch_pv_lat(const AttnArgs &a, cudaStream_t st) {
  switch (a.v.rice_k) {
    case 1: launch_pv_k<LAT, 1>(a, st); break;
    case 2: launch_pv_k<LAT, 2>(a, st); break;
    case 3: launch_pv_k<LAT, 3>(a, st); break;
    default: launch_pv_k<LAT, -1>(a, st); break;
  }
}

int launch_decode_qk(const QkArgs &a, int lattice, cudaStream_t st) {
  const int rows = a.B * a.Hq;
  rotate_queries_kernel<<<(rows + kRowThreads / 8 - 1) / (kRowThreads / 8), kRowThreads, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return 1;
  switch (lattice) {
    case 8: launch_qk_lat<8>(a, st); break;
    case 4: launch_qk_lat<4>(a, st); break;
    case 2: launch_qk_lat<2>(a, st); break;
    default: launch_qk_lat<1>(a, st); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_decode_attention(const AttnArgs &a, int k_lattice, int v_lattice, bool want_probs,
                            cudaStream_t st) {
  if (launch_decode_qk(a.qk, k_lattice, st) != 0) return 1;   // scores into a.qk.scores
  const unsigned rows = (unsigned)(a.qk.B * a.qk.Hq);
  switch (v_lattice) {
    case 8: launch_pv_lat<8>(a, st); break;
    case 4: launch_pv_lat<4>(a, st); break;
    case 2: launch_pv_lat<2>(a, st); break;
    default: launch_pv_lat<1>(a, st); break;
  }
  if (cudaGetLastError() != cudaSuccess) return 1;
  if (want_probs) {                              // the scores become probabilities in place
    softmax_kernel<<<rows, kSoftmaxThreads, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return 1;
  }
  return 0;
}

}  // namespace hq

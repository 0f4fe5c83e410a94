// hq_fused.cu -- kernels that consume compressed tiles without writing them
// out: attention scores from compressed K (hq_decode_qk), decode attention over
// compressed K and V (hq_decode_attention) and products with compressed
// weights (hq_decode_gemm) -- the summary's closing section, fused decode +
// MMA.  Each decodes only to the lattice domain e = v - u with the shared
// decoding step and moves the transform to the other operand: queries and
// activations are rotated once into that domain (q' = s_dec H D R q), and the
// attention output rows are transformed back once per row.
#include <cuda_runtime.h>

#include "hq_decode_lane.cuh"
#include "hq_umma.cuh"

namespace hq {

// q'[row] = s_dec * H * (D_h q[row]) for row = b * Hq + hq, h = hq / (Hq / n_kv).
__global__ void rotate_queries_kernel(QkArgs a) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= a.B * a.Hq) return;
  const int hq = row % a.Hq, h = hq / (a.Hq / a.n_kv);
  const int64_t seg = div_by((int64_t)h * a.n_tokens, a.dec.tiles_per_segment, a.dec.seg_shift);
  const uint32_t *mask = a.dec.signs + 4 * seg;
  float x[128];
  const uint16_t *q = a.q + (int64_t)row * kTile;
#pragma unroll
  for (int i = 0; i < 128; ++i) x[i] = __uint_as_float((uint32_t)q[i] << 16);
  if (a.dec.rot != nullptr) rotate128(a.dec.rot + seg * (int64_t)(kTile * kTile), x);
#pragma unroll
  for (int i = 0; i < 128; ++i)
    if ((mask[i >> 5] >> (i & 31)) & 1u) x[i] = -x[i];
  fwht128(x);
#pragma unroll
  for (int i = 0; i < 128; ++i) a.qrot[(int64_t)row * kTile + i] = __fmul_rn(x[i], a.dec.s_dec);
}

// Scores of one group of K tiles.  Lane r holds 16 lattice-domain values of
// its tile; partial dots with 8 query rows at a time are reduced over the
// tile's 8 lanes by a butterfly that leaves one finished row on each lane.
// The rotated query rows of the head of the group's first tile are staged in
// shared memory, laid out [row][lane r][16 + 4] so that the 8 lanes of a tile
// read distinct banks; tiles of another head read their rows from global.
constexpr int kQkRowsSmem = 64;
constexpr int kQkLaneStride = 20;                // 16 values + 4 floats of padding
constexpr int kQkEStride = kTile + 4;            // the group's e in the common case
template <int LAT, int K>
__global__ void __launch_bounds__(kDecThreads, 3)
scores_kernel(QkArgs a) {
  __shared__ uint64_t s_start[kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[2][kDecThreads / 32];
  __shared__ __align__(16) float s_q[kQkRowsSmem * 8 * kQkLaneStride];
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7;
  const int64_t g = blockIdx.x;
  const int G = a.Hq / a.n_kv;
  const int rows = a.B * G;                     // query rows that read one head
  const int h0 = (int)div_by(g * kGroupTiles, a.n_tokens, a.tok_shift);
  const bool staged = rows <= kQkRowsSmem;
  if (staged) {
    for (int i = tid; i < rows * 32; i += kDecThreads) {   // float4 units
      const int rr = i >> 5, c4 = i & 31;                   // row, 4-float chunk
      const int b = rr / G, gq = rr - b * G;
      const float4 v = __ldg(reinterpret_cast<const float4 *>(
          a.qrot + ((int64_t)b * a.Hq + (int64_t)h0 * G + gq) * kTile) + c4);
      const int rl = c4 >> 2, cc = (c4 & 3) * 4;
      *reinterpret_cast<float4 *>(&s_q[(rr * 8 + rl) * kQkLaneStride + cc]) = v;
    }
  }
  float e[16];
  const bool ok = decode_lane<LAT, K>(a.dec, g, e, s_start, s_warp);   // barriers inside
  if (!ok && tid == 0) atomicOr(a.dec.status, (uint32_t)HQ_ERR_CORRUPT);
  const int64_t tile = g * kGroupTiles + tl;
  const bool valid = tile < a.dec.n_tiles;
  const int h = valid ? (int)div_by(tile, a.n_tokens, a.tok_shift) : h0;
  const int64_t tok = valid ? tile - (int64_t)h * a.n_tokens : 0;
  const bool from_smem = staged && h == h0;
  // Common case: every query row staged and all 32 tiles tokens of head h0.
  // The group's e goes to shared memory and the 32 x rows block of scores is
  // a small product there: thread (tt, rq) computes tokens tt and tt + 16
  // for rows 4rq .. 4rq+3, each score one chain over d.
  const int64_t last = min(g * kGroupTiles + kGroupTiles, a.dec.n_tiles) - 1;
  if (staged && (int)div_by(last, a.n_tokens, a.tok_shift) == h0) {   // uniform
    __shared__ __align__(16) float s_et[kGroupTiles * kQkEStride];
    float4 *de = reinterpret_cast<float4 *>(&s_et[tl * kQkEStride + 16 * r]);
#pragma unroll
    for (int c = 0; c < 4; ++c) de[c] = make_float4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
    __syncthreads();
    const int tt = tid & 15, rq = tid >> 4;
    if (4 * rq < rows) {
      float acc[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = 0.0f;
      const int rlim = min(4, rows - 4 * rq);
#pragma unroll 2
      for (int k = 0; k < kTile; k += 4) {
        const float4 e0 = *reinterpret_cast<const float4 *>(&s_et[tt * kQkEStride + k]);
        const float4 e1 = *reinterpret_cast<const float4 *>(&s_et[(tt + 16) * kQkEStride + k]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 4 * rq + (i < rlim ? i : 0);
          const float4 qv = *reinterpret_cast<const float4 *>(
              &s_q[(rr * 8 + (k >> 4)) * kQkLaneStride + (k & 15)]);
          acc[i][0] = __fmaf_rn(qv.x, e0.x, acc[i][0]);
          acc[i][0] = __fmaf_rn(qv.y, e0.y, acc[i][0]);
          acc[i][0] = __fmaf_rn(qv.z, e0.z, acc[i][0]);
          acc[i][0] = __fmaf_rn(qv.w, e0.w, acc[i][0]);
          acc[i][1] = __fmaf_rn(qv.x, e1.x, acc[i][1]);
          acc[i][1] = __fmaf_rn(qv.y, e1.y, acc[i][1]);
          acc[i][1] = __fmaf_rn(qv.z, e1.z, acc[i][1]);
          acc[i][1] = __fmaf_rn(qv.w, e1.w, acc[i][1]);
        }
      }
      const int64_t t0 = g * kGroupTiles - (int64_t)h0 * a.n_tokens;   // token of tile 0
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i >= rlim) break;
        const int rr = 4 * rq + i, b = rr / G, gq = rr - b * G;
        float *dst = a.scores + ((int64_t)b * a.Hq + (int64_t)h0 * G + gq) * a.n_tokens + t0;
        if (g * kGroupTiles + tt < a.dec.n_tiles) dst[tt] = acc[i][0];
        if (g * kGroupTiles + tt + 16 < a.dec.n_tiles) dst[tt + 16] = acc[i][1];
      }
    }
    return;
  }
  for (int r0 = 0; r0 < rows; r0 += 8) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = r0 + i;
      float acc = 0.0f;
      if (rr < rows) {
        if (from_smem) {
          const float4 *qr = reinterpret_cast<const float4 *>(&s_q[(rr * 8 + r) * kQkLaneStride]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 qv = qr[c];
            acc = __fmaf_rn(qv.x, e[4 * c], acc);
            acc = __fmaf_rn(qv.y, e[4 * c + 1], acc);
            acc = __fmaf_rn(qv.z, e[4 * c + 2], acc);
            acc = __fmaf_rn(qv.w, e[4 * c + 3], acc);
          }
        } else {
          const int b = rr / G, gq = rr - b * G;
          const float4 *qr = reinterpret_cast<const float4 *>(
              a.qrot + ((int64_t)b * a.Hq + (int64_t)h * G + gq) * kTile + 16 * r);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 qv = __ldg(qr + c);
            acc = __fmaf_rn(qv.x, e[4 * c], acc);
            acc = __fmaf_rn(qv.y, e[4 * c + 1], acc);
            acc = __fmaf_rn(qv.z, e[4 * c + 2], acc);
            acc = __fmaf_rn(qv.w, e[4 * c + 3], acc);
          }
        }
      }
      p[i] = acc;
    }
    // reduce-scatter over the 8 lanes: after the step with mask m a lane keeps
    // the half of its slots whose bit m matches its own lane bit
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
#pragma unroll
      for (int i = 0; i < m; ++i) {
        const bool upper = (r & m) != 0;
        const float send = upper ? p[i] : p[i + m];
        const float keep = upper ? p[i + m] : p[i];
        const float got = __shfl_xor_sync(0xffffffffu, send, m);
        p[i] = __fadd_rn(keep, got);
      }
    }
    const int rr = r0 + r;                       // slot kept by lane r is row r0 + r
    if (valid && rr < rows) {
      const int b = rr / G, gq = rr - b * G;
      a.scores[((int64_t)b * a.Hq + (int64_t)h * G + gq) * a.n_tokens + tok] = p[0];
    }
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
// and column 64 + n holds (e_hi + e_lo) p_lo of row n, added once at the end.
// The block's 256 threads decode group g + 1 while the MMAs of group g run.
constexpr int kPvAKStride = 2304;                // bytes between K-cores of e^T (16 d-groups of 144)
constexpr int kPvAGStride = 144;                 // bytes between 8-dimension groups (16 B of padding)
constexpr int kPvBKStride = 144;                 // bytes between K-cores of B (16 B of padding)
constexpr int kPvBGStride = 1152;                // bytes between 8-row groups of B
constexpr int kPvOpBytes = 8 * kPvAKStride;      // 18432 per operand (e_hi^T, e_lo^T, B)
constexpr int kPvSmemBytes = 3 * kPvOpBytes;
constexpr uint32_t kPvIdesc = umma_idesc_tf32(128, 128);
constexpr uint32_t kPvTmemCols = 128;
constexpr uint32_t kPvWaitLimit = 1u << 22;

// This thread's 8 scaled scores z = fl(scale s) of group g (element
// i = tid + 256 k of the group's 64 rows x 32 tokens, row-major): consecutive
// threads read consecutive tokens of one row; tokens outside head h or rows
// past the end read as -inf (probability 0).
__device__ __forceinline__ void pv_load_z(const AttnArgs &a, int64_t g, int h, int row0, int G,
                                          int rows, int64_t tile_lo, int64_t tile_hi,
                                          float z[8]) {
  const int64_t T = a.qk.n_tokens;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = threadIdx.x + k * kDecThreads;
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
__global__ void __launch_bounds__(kDecThreads, 3) pv_kernel(AttnArgs a) {
  __shared__ uint64_t s_start[kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[2][kDecThreads / 32];
  __shared__ float s_m[kPvRows];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ uint32_t s_taddr;
  extern __shared__ __align__(128) unsigned char s_ops[];   // e_hi^T | e_lo^T | B
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7, warp = tid >> 5;
  const int chunk = blockIdx.x, h = blockIdx.y, rt = blockIdx.z;
  const int64_t T = a.qk.n_tokens;
  const int Hq = a.qk.Hq, G = Hq / a.qk.n_kv, rows = a.qk.B * G, row0 = rt * kPvRows;
  const int64_t tile_lo = (int64_t)h * T, tile_hi = tile_lo + T;
  const int64_t g_first = tile_lo / kGroupTiles, g_end = (tile_hi - 1) / kGroupTiles + 1;
  const int64_t gb = g_first + (int64_t)chunk * kPvGroupsPerChunk;
  const int64_t ge = min(gb + (int64_t)kPvGroupsPerChunk, g_end);
  if (warp == 0) tmem_alloc(&s_taddr, kPvTmemCols);
  if (tid == 32) mbar_init(&s_bar, 1);
  // this chunk's softmax statistics per row: m = max z over its tokens and
  // l = sum exp(z - m) (four threads per row, then a fixed shuffle tree)
  {
    const int rr = tid >> 2, q = tid & 3, row = row0 + rr;
    const int64_t c_lo = max(gb * kGroupTiles, tile_lo), c_hi = min(ge * kGroupTiles, tile_hi);
    const float *srow = nullptr;
    if (row < rows) {
      const int b = row / G, gq = row - b * G;
      srow = a.qk.scores + ((int64_t)b * Hq + (int64_t)h * G + gq) * T - tile_lo;
    }
    float m = -INFINITY, l = 0.0f;
    if (srow != nullptr)
      for (int64_t t = c_lo + q; t < c_hi; t += 4) m = fmaxf(m, __fmul_rn(srow[t], a.scale));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    if (srow != nullptr && m != -INFINITY)
      for (int64_t t = c_lo + q; t < c_hi; t += 4)
        l = __fadd_rn(l, expf(__fsub_rn(__fmul_rn(srow[t], a.scale), m)));
    l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, 1));
    l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, 2));
    if (q == 0) {
      s_m[rr] = m;
      a.stats[(((int64_t)h * a.chunks + chunk) * a.rowtiles + rt) * kPvRows + rr] = make_float2(m, l);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = s_taddr;
  const uint32_t a_hi = smem_addr(s_ops), a_lo = a_hi + kPvOpBytes, b_op = a_hi + 2 * kPvOpBytes;
  // this thread's slots: e^T (d = 16 r + c, token tl) and B (row i >> 5, token i & 31)
  float *const ehi = reinterpret_cast<float *>(s_ops) +
                     (288 * r + (tl >> 2) * kPvAKStride + (tl & 3) * 4) / 4;
  float *const elo = ehi + kPvOpBytes / 4;
  float *const bp = reinterpret_cast<float *>(s_ops + 2 * kPvOpBytes) +
                    ((tid >> 5) * 16 + ((tid & 31) >> 2) * kPvBKStride + (tid & 3) * 4) / 4;
  bool ok_wait = true;                           // block-uniform
  int committed = 0;                             // groups whose MMAs were issued
  // the scores of a group are loaded one group ahead, so that their latency
  // hides behind the decoding of the current one
  float pn[8];
  if (gb < ge) pv_load_z(a, gb, h, row0, G, rows, tile_lo, tile_hi, pn);
  for (int64_t g = gb; g < ge; ++g) {            // block-uniform bounds
    const int i = (int)(g - gb);
    float e[16];
    const bool ok = decode_lane<LAT, K>(a.v, g, e, s_start, s_warp);   // barriers inside
    if (!ok && tid == 0) atomicOr(a.v.status, (uint32_t)HQ_ERR_CORRUPT);
    // the MMAs of the previous group must be done with the operands
    if (i > 0 && ok_wait) ok_wait = mbar_wait(&s_bar, (uint32_t)(i - 1) & 1u, kPvWaitLimit);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float hi, lo;
      split_tf32(e[c], hi, lo);
      const int off = ((c >> 3) * kPvAGStride + (c & 7) * 16) / 4;
      ehi[off] = hi;
      elo[off] = lo;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {                // p = exp(z - m), 0 for z = -inf
      const float mm = s_m[(tid >> 5) + 8 * k];
      const float p = pn[k] == -INFINITY ? 0.0f : expf(__fsub_rn(pn[k], mm));
      float hi, lo;
      split_tf32(p, hi, lo);
      bp[k * kPvBGStride / 4] = hi;              // rows (tid >> 5) + 8 k
      bp[(k + 8) * kPvBGStride / 4] = lo;        // rows 64 + (tid >> 5) + 8 k
    }
    if (g + 1 < ge) pv_load_z(a, g + 1, h, row0, G, rows, tile_lo, tile_hi, pn);
    fence_async_smem();
    ok_wait = __syncthreads_and(ok_wait) != 0;
    if (!ok_wait) continue;
    ++committed;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_tf32(taddr, umma_desc(a_hi + ks * 2 * kPvAKStride, kPvAKStride, kPvAGStride),
                  umma_desc(b_op + ks * 2 * kPvBKStride, kPvBKStride, kPvBGStride), kPvIdesc,
                  (i > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_tf32(taddr, umma_desc(a_lo + ks * 2 * kPvAKStride, kPvAKStride, kPvAGStride),
                  umma_desc(b_op + ks * 2 * kPvBKStride, kPvBKStride, kPvBGStride), kPvIdesc, 1u);
      umma_commit(&s_bar);
    }
  }
  if (committed > 0) {
    if (ok_wait) ok_wait = mbar_wait(&s_bar, (uint32_t)(committed - 1) & 1u, kPvWaitLimit);
    ok_wait = __syncthreads_and(ok_wait) != 0;
    if (ok_wait) {
      tc_fence_after();
      // warp w reads dimensions 32 (w % 4) + lane for rows 32 (w / 4) .. +31
      const int qd = warp & 3, hf = warp >> 2, d = 32 * qd + (tid & 31);
      float *part = a.partials +
                    ((((int64_t)h * a.chunks + chunk) * a.rowtiles + rt) * kPvRows) * kTile;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float vh[16], vl[16];
        const uint32_t lane_addr = taddr + ((uint32_t)(32 * qd) << 16);
        tmem_ld16(lane_addr + (uint32_t)(32 * hf + 16 * jj), vh);
        tmem_ld16(lane_addr + (uint32_t)(64 + 32 * hf + 16 * jj), vl);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          part[(int64_t)(32 * hf + 16 * jj + j) * kTile + d] = __fadd_rn(vh[j], vl[j]);
      }
    }
  }
  if (!ok_wait) {
    if (tid == 0) atomicOr(a.v.status, (uint32_t)HQ_ERR_TIMEOUT);
    // the operands' last MMAs may still be in flight: give them a bounded
    // while before the tensor memory goes back
    if (committed > 0) mbar_wait(&s_bar, (uint32_t)(committed - 1) & 1u, kPvWaitLimit);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(taddr, kPvTmemCols);
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

// ---------------------------------------------------------------- weights
// x'[b][j] = s_dec * H * (D x[b][j]) for each 128-column tile j of activation
// row b (the whole matrix is one sign segment).
__global__ void rotate_x_kernel(GemmArgs a) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // (b, j)
  if (i >= (int64_t)a.B * a.tpr) return;
  const uint32_t *mask = a.dec.signs;
  float x[128];
  const uint16_t *src = a.x + i * kTile;
#pragma unroll
  for (int k = 0; k < 128; ++k) x[k] = __uint_as_float((uint32_t)src[k] << 16);
  if (a.dec.rot != nullptr) rotate128(a.dec.rot, x);      // the matrix is one segment
#pragma unroll
  for (int k = 0; k < 128; ++k)
    if ((mask[k >> 5] >> (k & 31)) & 1u) x[k] = -x[k];
  fwht128(x);
#pragma unroll
  for (int k = 0; k < 128; ++k) a.xrot[i * kTile + k] = __fmul_rn(x[k], a.dec.s_dec);
}

// Each tile's share of y: lane r of tile t holds 16 lattice-domain values;
// partial dots with 8 activation rows at a time are reduced over the tile's
// 8 lanes by a butterfly that leaves one finished row on each lane.
template <int LAT, int K>
__global__ void __launch_bounds__(kDecThreads, 3) gemm_kernel(GemmArgs a) {
  __shared__ uint64_t s_start[kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[2][kDecThreads / 32];
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7;
  const int64_t g = blockIdx.x;
  float e[16];
  const bool ok = decode_lane<LAT, K>(a.dec, g, e, s_start, s_warp);   // barriers inside
  if (!ok && tid == 0) atomicOr(a.dec.status, (uint32_t)HQ_ERR_CORRUPT);
  const int64_t tile = g * kGroupTiles + tl;
  const bool valid = tile < a.dec.n_tiles;
  const int64_t row = valid ? div_by(tile, a.tpr, a.tpr_shift) : 0;
  const int64_t j = valid ? tile - row * a.tpr : 0;
  for (int b0 = 0; b0 < a.B; b0 += 8) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float acc = 0.0f;
      if (b0 + i < a.B) {
        const float4 *xr = reinterpret_cast<const float4 *>(
            a.xrot + (int64_t)(b0 + i) * a.cols + j * kTile + 16 * r);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 xv = __ldg(xr + c);
          acc = __fmaf_rn(xv.x, e[4 * c], acc);
          acc = __fmaf_rn(xv.y, e[4 * c + 1], acc);
          acc = __fmaf_rn(xv.z, e[4 * c + 2], acc);
          acc = __fmaf_rn(xv.w, e[4 * c + 3], acc);
        }
      }
      p[i] = acc;
    }
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
#pragma unroll
      for (int i = 0; i < m; ++i) {
        const bool upper = (r & m) != 0;
        const float send = upper ? p[i] : p[i + m];
        const float keep = upper ? p[i + m] : p[i];
        const float got = __shfl_xor_sync(0xffffffffu, send, m);
        p[i] = __fadd_rn(keep, got);
      }
    }
    const int b = b0 + r;                        // slot kept by lane r is row b0 + r
    if (valid && b < a.B) a.partial[(int64_t)b * a.dec.n_tiles + tile] = p[0];
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

template <int LAT>
static void launch_qk_lat(const QkArgs &a, cudaStream_t st) {
  dim3 grid((unsigned)a.dec.n_groups), block(kDecThreads);
  switch (a.dec.rice_k) {
    case 1: scores_kernel<LAT, 1><<<grid, block, 0, st>>>(a); break;
    case 2: scores_kernel<LAT, 2><<<grid, block, 0, st>>>(a); break;
    case 3: scores_kernel<LAT, 3><<<grid, block, 0, st>>>(a); break;
    default: scores_kernel<LAT, -1><<<grid, block, 0, st>>>(a); break;
  }
}

template <int LAT, int K>
static void launch_pv_one(const AttnArgs &a, dim3 grid, dim3 block, cudaStream_t st) {
  cudaFuncSetAttribute(pv_kernel<LAT, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPvSmemBytes);
  pv_kernel<LAT, K><<<grid, block, kPvSmemBytes, st>>>(a);
}

template <int LAT>
static void launch_pv_lat(const AttnArgs &a, cudaStream_t st) {
  dim3 grid((unsigned)a.chunks, (unsigned)a.qk.n_kv, (unsigned)a.rowtiles), block(kDecThreads);
  switch (a.v.rice_k) {
    case 1: launch_pv_one<LAT, 1>(a, grid, block, st); break;
    case 2: launch_pv_one<LAT, 2>(a, grid, block, st); break;
    case 3: launch_pv_one<LAT, 3>(a, grid, block, st); break;
    default: launch_pv_one<LAT, -1>(a, grid, block, st); break;
  }
}

template <int LAT>
static void launch_gemm_lat(const GemmArgs &a, cudaStream_t st) {
  dim3 grid((unsigned)a.dec.n_groups), block(kDecThreads);
  switch (a.dec.rice_k) {
    case 2: gemm_kernel<LAT, 2><<<grid, block, 0, st>>>(a); break;
    case 3: gemm_kernel<LAT, 3><<<grid, block, 0, st>>>(a); break;
    case 4: gemm_kernel<LAT, 4><<<grid, block, 0, st>>>(a); break;
    default: gemm_kernel<LAT, -1><<<grid, block, 0, st>>>(a); break;
  }
}

int launch_decode_qk(const QkArgs &a, int lattice, cudaStream_t st) {
  const int rows = a.B * a.Hq;
  rotate_queries_kernel<<<(rows + 127) / 128, 128, 0, st>>>(a);
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
  pv_finish_kernel<<<rows, kTile, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return 1;
  if (want_probs) {                              // the scores become probabilities in place
    softmax_kernel<<<rows, kSoftmaxThreads, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return 1;
  }
  return 0;
}

int launch_decode_gemm(const GemmArgs &a, int lattice, cudaStream_t st) {
  const int64_t xt = (int64_t)a.B * a.tpr;
  rotate_x_kernel<<<(unsigned)((xt + 127) / 128), 128, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return 1;
  switch (lattice) {
    case 8: launch_gemm_lat<8>(a, st); break;
    case 4: launch_gemm_lat<4>(a, st); break;
    case 2: launch_gemm_lat<2>(a, st); break;
    default: launch_gemm_lat<1>(a, st); break;
  }
  if (cudaGetLastError() != cudaSuccess) return 1;
  const int64_t warps = (int64_t)a.B * a.rows;
  gemm_reduce_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace hq

// hq_decode.cu -- decoder and fused score kernel of the HyperQuant tile codec.
//
// A block of 256 threads decodes one index group of 32 tiles; lane r of a
// tile handles symbols 16r .. 16r+15 (two 8-vectors).  The block finds where
// every lane's unary codes start by a block-wide popcount scan of the U-area
// (every one bit there ends a symbol: 16 per lane).  Each lane reads its remainders at their fixed
// position and its unary codes with count-leading-zeros, restores the
// stripped bits, regenerates the dither and inverts the transform
// (HyperQuant summary, Method 1-4 in reverse); outputs are stored with
// contiguous 32-byte (bf16) / 64-byte (fp32) writes per lane.  Every loop is
// bounded by the group's word count from the index, and a group that fails
// any check is written as zeros with HQ_ERR_CORRUPT.
//
// hq_decode_qk (the summary's closing section, fused decode + MMA) decodes K
// only to the lattice domain e = v - u and dots it with queries rotated once
// into that domain, q' = s_dec H D q, so K is never written and no inverse
// transform is run per key.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hq_device.cuh"
#include "hq_internal.h"

namespace hq {

constexpr int kDecThreads = 256;

// nb (1..64) bits starting at bit `pos` of W, MSB-first, right-aligned.
__device__ __forceinline__ uint64_t read_bits(const uint32_t *W, uint64_t pos, int nb) {
  const uint64_t w = pos >> 5;
  const int sh = (int)(pos & 31);
  const int need = (sh + nb + 31) >> 5;         // words touched (1..3)
  const uint32_t a0 = W[w];
  const uint32_t a1 = need > 1 ? W[w + 1] : 0u;
  const uint32_t a2 = need > 2 ? W[w + 2] : 0u;
  const uint64_t hi = ((uint64_t)a0 << 32) | a1;
  const uint64_t v = (hi << sh) | (sh ? ((uint64_t)a2 >> (32 - sh)) : 0ull);
  return nb >= 64 ? v : (v >> (64 - nb));
}

// MSB-first position (0..31) of the n-th (1-based, n <= popc(x)) set bit of
// x: a branch-free binary search on population counts.
__device__ __forceinline__ int nth_set_bit_msb(uint32_t x, int n) {
  int p = 0;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const int c = __popc(x >> (32 - w));        // ones among the top w bits
    const bool skip = c < n;
    n -= skip ? c : 0;
    x = skip ? (x << w) : x;
    p += skip ? w : 0;
  }
  return p;
}


// Quotients of 8 unary codes from bit pos in the general case (a code longer
// than the lane's 64-bit window, or a quotient of 32 or more): one 32-bit view
// per step, runs of zeros counted 32 at a time.  Lanes rarely take it (a
// divergent branch).  next = the bit after the 8th code; bad = a quotient
// above qmax or codes running past the group's last word.
template <class P>
struct Quot8 {
  uint32_t q[8];
  P next;
  bool bad;
};

template <class P>
__device__ __forceinline__ Quot8<P> unary8_general(const uint32_t *W, P pos, P nwords, int k) {
  Quot8<P> out;
  out.bad = false;
  const uint32_t qmax = (kSymbolLimit - 1u) >> k;
  const P end = nwords * 32;
  for (int j = 0; j < 8; ++j) out.q[j] = 0u;
  for (int j = 0; j < 8 && !out.bad; ++j) {
    uint32_t q = 0;
    for (;;) {
      if (pos >= end || q > qmax) { out.bad = true; break; }
      const P w = pos >> 5;
      const uint32_t b0 = __ldg(W + w), b1 = w + 1 < nwords ? __ldg(W + w + 1) : 0u;
      const uint32_t view = __funnelshift_l(b1, b0, (uint32_t)(pos & 31));
      if (view == 0u) {                          // 32 more zeros of this code
        q += 32u;
        pos += 32;
        continue;
      }
      const uint32_t z = __clz(view);
      q += z;
      pos += (P)(z + 1u);
      break;
    }
    if (q > qmax) out.bad = true;
    out.q[j] = q;
  }
  out.next = pos;
  return out;
}

// Finds where every lane's unary codes start, parses this lane's 16 symbols
// and returns e = v - u for them (lattice domain).  The group's words are read
// straight from global memory (each is read by the scan first, so the parse
// hits L1).  Bit positions within the group have type P: 32-bit for groups
// below 2^31 bits (every group of a sane stream), 64-bit otherwise.  The
// return value is block-uniform: false when the group is corrupt (e is then
// all zeros).
template <int LAT, int K, class P>
__device__ __forceinline__ bool decode_lane_p(const DecodeArgs &a, int64_t g, int nt,
                                              const uint32_t *W, P nwords, bool bad,
                                              float e[16], P *s_start,
                                              uint32_t (*s_warp)[kDecThreads / 32]) {
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7, lane = tid & 31, warp = tid >> 5;
  const int k = K >= 0 ? K : a.rice_k;
  const P R = (P)(K >= 0 ? tile_rbits<LAT>(K) : a.rbits);
  const P ustart = (P)nt * R;
  if (ustart > nwords * 32) bad = true;

  // ---- unary starts: the 16m-th one of the U-area ends lane m-1's codes.
  // One word per thread per window; a warp scan plus one barrier per window.
  const P want = (P)128 * (P)nt;
  P ones = 0;
  if (!bad) {
    int par = 0;
    for (P wb = ustart >> 5; wb < nwords; wb += kDecThreads) {
      const P w = wb + (P)tid;
      const bool wact = wb + (P)(warp * 32) < nwords;   // warp-uniform: any word to scan
      uint32_t word = 0u, pc = 0u, incl = 0u;
      if (wact) {
        word = w < nwords ? __ldg(W + w) : 0u;
        if (w == (ustart >> 5)) word &= 0xFFFFFFFFu >> (ustart & 31);
        pc = __popc(word);
        incl = pc;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += o;
        }
      }
      if (lane == 31) s_warp[par][warp] = incl;
      __syncthreads();
      static_assert(kDecThreads / 32 == 8, "two 16-byte reads of the warp totals");
      const uint4 q0 = reinterpret_cast<const uint4 *>(s_warp[par])[0];
      const uint4 q1 = reinterpret_cast<const uint4 *>(s_warp[par])[1];
      const uint32_t ws[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      uint32_t before_w = 0, total = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        before_w += i < warp ? ws[i] : 0u;
        total += ws[i];
      }
      if (wact) {
        const P before = ones + (P)(before_w + incl - pc);
        P m = (before / 16 + 1) * 16;             // at most two boundaries per word
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
          if (m <= before + pc && m <= want)
            s_start[m / 16] = w * 32 + (P)nth_set_bit_msb(word, (int)(m - before)) + 1;
          m += 16;
        }
      }
      ones += total;
      par ^= 1;
    }
  }
  if (tid == 0) s_start[0] = ustart;
  __syncthreads();
  if (!bad && (ones != want || ((s_start[8 * nt] + 31) >> 5) != nwords)) bad = true;

  // ---- this lane's symbols: remainder bits first, then the quotients
  bool lbad = false;
  const bool valid = tl < nt;
  const int rb8 = K >= 0 ? rbits8<LAT>(K) : (int)(R / 16);
  const P rpos = (P)tl * R + (P)(r * 2 * rb8);
  uint64_t rv[2] = {0ull, 0ull};                 // remainder bits of each 8-group
  uint32_t qp[4] = {0u, 0u, 0u, 0u};             // quotient j in byte j % 4 of qp[j / 4]
  bool slow = false;
  P pos = 0, stop = 0;
  if (!bad && valid) {
    if (K >= 0 && rb8 > 0) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) rv[jj] = read_bits(W, (uint64_t)(rpos + (P)(jj * rb8)), rb8);
    }
    pos = s_start[tid];
    stop = s_start[tid + 1];
    slow = stop - pos > (P)64;
    if (!slow) {
      // The lane's 16 codes (exactly 16 ones, the last at bit stop-1) lie in
      // the 64 bits (hi:lo) from pos: each quotient is the count of zeros
      // before the next one.  A quotient of 32 or more (hi all zeros) leaves
      // bit 5 set in zo and the lane takes the general parser; shorter
      // quotients are below qmax for every k <= 15, and the 16th one ends at
      // stop by construction of the boundaries.
      const P pw = pos >> 5;
      const uint32_t a0 = pw < nwords ? __ldg(W + pw) : 0u;
      const uint32_t a1 = pw + 1 < nwords ? __ldg(W + pw + 1) : 0u;
      const uint32_t a2 = pw + 2 < nwords ? __ldg(W + pw + 2) : 0u;
      const uint32_t sh = (uint32_t)(pos & 31);
      uint32_t hi = __funnelshift_l(a1, a0, sh), lo = __funnelshift_l(a2, a1, sh);
      uint32_t zo = 0u;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t z = __clz(hi);
        zo |= z;
        qp[j >> 2] += z << (8 * (j & 3));
        hi = __funnelshift_lc(lo, hi, z + 1u);
        lo = shl_clamp(lo, z + 1u);
      }
      slow = (zo & 32u) != 0u;
    }
  }

  // ---- symbols, restore stripped bits, subtract the dither
  if (!bad && valid) {
    const uint64_t gt = a.tile_base + (uint64_t)(g * kGroupTiles + tl);
    P posj = pos;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      uint32_t s8[8];
      if (K >= 0) {
        constexpr int KK = K >= 0 ? K : 0;
        int off = rb8;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int lowb = stripped_low_bits<LAT>(c, KK);
          const int nb = KK - lowb;
          off -= nb;
          s8[c] = nb > 0 ? (uint32_t)((rv[jj] >> off) & ((1ull << nb) - 1ull)) << lowb : 0u;
        }
      } else {
        P q = rpos + (P)(jj * rb8);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int lowb = stripped_low_bits<LAT>(c, k);
          const int nb = k - lowb;
          s8[c] = nb > 0 ? (uint32_t)read_bits(W, (uint64_t)q, nb) << lowb : 0u;
          q += (P)(nb > 0 ? nb : 0);
        }
      }
      if (!slow) {
#pragma unroll
        for (int c = 0; c < 8; ++c) s8[c] += ((qp[2 * jj + (c >> 2)] >> (8 * (c & 3))) & 0xFFu) << k;
      } else {
        const Quot8<P> g8 = unary8_general<P>(W, posj, nwords, k);
        posj = g8.next;
        lbad |= g8.bad;
#pragma unroll
        for (int c = 0; c < 8; ++c) s8[c] += g8.q[c] << k;
      }
      int32_t v[8];
      unfold8<LAT>(s8, k, v, &lbad);
      float u[8];
      if (a.dither) {
        dither8<LAT>(a.keys, gt, (uint32_t)(2 * r + jj), u);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) u[i] = 0.0f;
      }
      float fv[8];
      point8<LAT>(v, fv);
#pragma unroll
      for (int i = 0; i < 8; ++i) e[8 * jj + i] = __fsub_rn(fv[i], u[i]);
    }
    if (slow && posj != stop) lbad = true;       // bit after the last code
  }
  const int any_bad = __syncthreads_or((bad || lbad) ? 1 : 0);
  if (any_bad || !valid) {
#pragma unroll
    for (int i = 0; i < 16; ++i) e[i] = 0.0f;
  }
  return !any_bad;
}

// Dispatch on the group's size: 32-bit bit positions unless the group holds
// 2^31 bits or more.
template <int LAT, int K>
__device__ __forceinline__ bool decode_lane(const DecodeArgs &a, int64_t g, float e[16],
                                            uint64_t *s_start64,
                                            uint32_t (*s_warp)[kDecThreads / 32]) {
  const int64_t t0 = g * kGroupTiles;
  const int nt = (int)min((int64_t)kGroupTiles, a.n_tiles - t0);
  const uint64_t base = a.offsets[g], end = a.offsets[g + 1];
  const bool bad = end < base || end > a.stream_words;
  const uint64_t nwords = bad ? 0 : end - base;
  const uint32_t *W = a.stream + (bad ? 0 : base);
  if (nwords < (1ull << 26))
    return decode_lane_p<LAT, K, uint32_t>(a, g, nt, W, (uint32_t)nwords, bad, e,
                                           reinterpret_cast<uint32_t *>(s_start64), s_warp);
  return decode_lane_p<LAT, K, uint64_t>(a, g, nt, W, nwords, bad, e, s_start64, s_warp);
}

template <int LAT, int K>
__global__ void __launch_bounds__(kDecThreads, 8)
decode_kernel(DecodeArgs a) {
  __shared__ uint64_t s_start[kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[2][kDecThreads / 32];
  __shared__ float4 s_scale[kTile / 4];          // D_i * s_dec of the block's first segment
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7;
  const int64_t g = blockIdx.x;
  const int64_t seg0 = div_by(g * kGroupTiles, a.tiles_per_segment, a.seg_shift);
  if (tid < kTile) {
    const uint32_t mword = __ldg(a.signs + 4 * seg0 + (tid >> 5));
    reinterpret_cast<float *>(s_scale)[tid] =
        __uint_as_float(__float_as_uint(a.s_dec) ^ (((mword >> (tid & 31)) & 1u) << 31));
  }
  float e[16];
  const bool ok = decode_lane<LAT, K>(a, g, e, s_start, s_warp);
  const int64_t t = g * kGroupTiles + tl;
  if (!ok && tid == 0) atomicOr(a.status, (uint32_t)HQ_ERR_CORRUPT);
  // the transform runs on every lane of the block (shuffles need full warps)
  fwht128_x8(e, r);
  const bool tvalid = t < a.n_tiles;
  if (a.rot == nullptr && !tvalid) return;
  if (ok && tvalid) {
    // x = D fl(z s_dec) = fl(z (D s_dec)): the sign commutes with rounding
    if (div_by(t, a.tiles_per_segment, a.seg_shift) == seg0) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 sc = s_scale[4 * r + c];
        e[4 * c] = __fmul_rn(e[4 * c], sc.x);
        e[4 * c + 1] = __fmul_rn(e[4 * c + 1], sc.y);
        e[4 * c + 2] = __fmul_rn(e[4 * c + 2], sc.z);
        e[4 * c + 3] = __fmul_rn(e[4 * c + 3], sc.w);
      }
    } else {
      const uint32_t *mask = a.signs + 4 * (div_by(t, a.tiles_per_segment, a.seg_shift));
      const uint32_t mw = __ldg(mask + (r >> 1)) >> (16 * (r & 1));
#pragma unroll
      for (int i = 0; i < 16; ++i)
        e[i] = __fmul_rn(e[i], __uint_as_float(__float_as_uint(a.s_dec) ^ (((mw >> i) & 1u) << 31)));
    }
  }
  if (a.rot != nullptr) {                        // uniform: x_hat = R^T y, chains over i
    // [32 tiles x 128] x [128 x 128] in shared memory: y transposed [128][36]
    // (later reused for the result [32][132]) and R row-major [128][132]
    constexpr int kYS = kGroupTiles + 4, kRS = kTile + 4;
    extern __shared__ __align__(16) float s_dyn[];
    float *s_yt = s_dyn;
    float *s_r = s_dyn + kTile * kYS;
#pragma unroll
    for (int c = 0; c < 16; ++c) s_yt[(16 * r + c) * kYS + tl] = e[c];
    const float4 *R4 = reinterpret_cast<const float4 *>(a.rot + seg0 * (int64_t)(kTile * kTile));
    for (int idx = tid; idx < kTile * kTile / 4; idx += kDecThreads)
      *reinterpret_cast<float4 *>(s_r + (idx >> 5) * kRS + 4 * (idx & 31)) = __ldg(R4 + idx);
    __syncthreads();
    const int tb = tid >> 5, ob = tid & 31;     // tiles 4tb.., outputs 4ob..
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[u][c] = 0.0f;
#pragma unroll 4
    for (int i = 0; i < kTile; ++i) {
      const float4 yv = *reinterpret_cast<const float4 *>(s_yt + i * kYS + 4 * tb);
      const float4 rv = *reinterpret_cast<const float4 *>(s_r + i * kRS + 4 * ob);
      const float ys[4] = {yv.x, yv.y, yv.z, yv.w}, rs[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[u][c] = __fmaf_rn(rs[c], ys[u], acc[u][c]);
    }
    __syncthreads();
    float *s_o = s_dyn;                          // [32][132]
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<float4 *>(s_o + (4 * tb + u) * kRS + 4 * ob) =
          make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 q = *reinterpret_cast<const float4 *>(s_o + tl * kRS + 16 * r + 4 * c);
      e[4 * c] = q.x;
      e[4 * c + 1] = q.y;
      e[4 * c + 2] = q.z;
      e[4 * c + 3] = q.w;
    }
    if (!tvalid) return;
  }
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
// Softmax over the tokens of one query row, in place: p = exp(z - m) / l with
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

// Partial sums P . E of one KV head over a chunk of its token groups, in the
// lattice domain: V's tiles are decoded only to e = v - u (no inverse
// transform per token), since sum_t p_t Vhat_t = D s_dec H (sum_t p_t e_t)
// up to rounding; pv_finish_kernel applies H, s_dec and D once per query
// row.  The group's e (32 tokens x 128) and probabilities (32 tokens x 64
// rows) are staged in shared memory; thread (rb, db) accumulates rows
// 4rb..4rb+3 x dims 8db..8db+7 over all tokens of the chunk.  Tokens of the
// group outside head h (a group that straddles two heads) get p = 0.
constexpr int kPvEStride = kTile + 4;
constexpr int kPvPStride = kPvRows + 4;
template <int LAT, int K>
__global__ void __launch_bounds__(kDecThreads, 2) pv_kernel(AttnArgs a) {
  __shared__ uint64_t s_start[kDecThreads + 1];
  __shared__ __align__(16) uint32_t s_warp[2][kDecThreads / 32];
  __shared__ __align__(16) float s_e[kGroupTiles * kPvEStride];
  __shared__ __align__(16) float s_p[kGroupTiles * kPvPStride];
  const int tid = threadIdx.x, tl = tid >> 3, r = tid & 7;
  const int chunk = blockIdx.x, h = blockIdx.y, rt = blockIdx.z;
  const int64_t T = a.qk.n_tokens;
  const int Hq = a.qk.Hq, G = Hq / a.qk.n_kv, rows = a.qk.B * G, row0 = rt * kPvRows;
  const int64_t tile_lo = (int64_t)h * T, tile_hi = tile_lo + T;
  const int64_t g_first = tile_lo / kGroupTiles, g_end = (tile_hi - 1) / kGroupTiles + 1;
  const int64_t gb = g_first + (int64_t)chunk * kPvGroupsPerChunk;
  const int64_t ge = min(gb + (int64_t)kPvGroupsPerChunk, g_end);
  const int rb = tid >> 4, db = tid & 15;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
  for (int64_t g = gb; g < ge; ++g) {            // block-uniform bounds
    float e[16];
    const bool ok = decode_lane<LAT, K>(a.v, g, e, s_start, s_warp);   // barriers inside
    if (!ok && tid == 0) atomicOr(a.v.status, (uint32_t)HQ_ERR_CORRUPT);
    float4 *de = reinterpret_cast<float4 *>(&s_e[tl * kPvEStride + 16 * r]);
#pragma unroll
    for (int c = 0; c < 4; ++c) de[c] = make_float4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
    // probabilities: consecutive threads read consecutive tokens of one row
    for (int i = tid; i < kGroupTiles * kPvRows; i += kDecThreads) {
      const int rr = i >> 5, j = i & 31;
      const int64_t tile = g * kGroupTiles + j;
      const int row = row0 + rr;
      float pv = 0.0f;
      if (tile >= tile_lo && tile < tile_hi && row < rows) {
        const int b = row / G, gq = row - b * G;
        pv = a.qk.scores[((int64_t)b * Hq + (int64_t)h * G + gq) * T + (tile - tile_lo)];
      }
      s_p[j * kPvPStride + rr] = pv;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kGroupTiles; ++j) {
      const float4 pj = *reinterpret_cast<const float4 *>(&s_p[j * kPvPStride + 4 * rb]);
      const float4 e0 = *reinterpret_cast<const float4 *>(&s_e[j * kPvEStride + 8 * db]);
      const float4 e1 = *reinterpret_cast<const float4 *>(&s_e[j * kPvEStride + 8 * db + 4]);
      const float pr[4] = {pj.x, pj.y, pj.z, pj.w};
      const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[i][c] = __fmaf_rn(pr[i], ev[c], acc[i][c]);
    }
    __syncthreads();
  }
  float *part = a.partials +
                ((((int64_t)h * a.chunks + chunk) * a.rowtiles + rt) * kPvRows) * kTile;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 *dst = reinterpret_cast<float4 *>(part + (int64_t)(4 * rb + i) * kTile + 8 * db);
    dst[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    dst[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

// out[b][hq] = D_h * fl(H (sum over chunks of the partial rows) * s_dec), the
// chunks summed in order; one block of 128 threads per query row.
__global__ void __launch_bounds__(kTile) pv_finish_kernel(AttnArgs a) {
  __shared__ float x[kTile];
  const int row = blockIdx.x, d = threadIdx.x;
  const int Hq = a.qk.Hq, G = Hq / a.qk.n_kv;
  const int b = row / Hq, hq = row - b * Hq, h = hq / G;
  const int rr = b * G + (hq - h * G), rt = rr / kPvRows, rl = rr - rt * kPvRows;
  float s = 0.0f;
  for (int c = 0; c < a.chunks; ++c)
    s = __fadd_rn(s, a.partials[((((int64_t)h * a.chunks + c) * a.rowtiles + rt) * kPvRows + rl) *
                                    kTile + d]);
  x[d] = s;
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

constexpr size_t kDecRotSmemBytes = (size_t)(kTile * (kGroupTiles + 4) + kTile * (kTile + 4)) * 4;

template <int LAT, int K>
static void launch_dec_one(const DecodeArgs &a, cudaStream_t st) {
  const size_t dyn = a.rot != nullptr ? kDecRotSmemBytes : 0;
  if (dyn)
    cudaFuncSetAttribute(decode_kernel<LAT, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)dyn);
  decode_kernel<LAT, K><<<dim3((unsigned)a.n_groups), dim3(kDecThreads), dyn, st>>>(a);
}

template <int LAT>
static void launch_dec_lat(const DecodeArgs &a, cudaStream_t st) {
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

template <int LAT>
static void launch_pv_lat(const AttnArgs &a, cudaStream_t st) {
  dim3 grid((unsigned)a.chunks, (unsigned)a.qk.n_kv, (unsigned)a.rowtiles), block(kDecThreads);
  switch (a.v.rice_k) {
    case 1: pv_kernel<LAT, 1><<<grid, block, 0, st>>>(a); break;
    case 2: pv_kernel<LAT, 2><<<grid, block, 0, st>>>(a); break;
    case 3: pv_kernel<LAT, 3><<<grid, block, 0, st>>>(a); break;
    default: pv_kernel<LAT, -1><<<grid, block, 0, st>>>(a); break;
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

int launch_decode(const DecodeArgs &a, int lattice, cudaStream_t st) {
  switch (lattice) {
    case 8: launch_dec_lat<8>(a, st); break;
    case 4: launch_dec_lat<4>(a, st); break;
    case 2: launch_dec_lat<2>(a, st); break;
    default: launch_dec_lat<1>(a, st); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
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

int launch_decode_attention(const AttnArgs &a, int k_lattice, int v_lattice, cudaStream_t st) {
  if (launch_decode_qk(a.qk, k_lattice, st) != 0) return 1;   // scores into a.qk.scores
  const unsigned rows = (unsigned)(a.qk.B * a.qk.Hq);
  softmax_kernel<<<rows, kSoftmaxThreads, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return 1;
  switch (v_lattice) {
    case 8: launch_pv_lat<8>(a, st); break;
    case 4: launch_pv_lat<4>(a, st); break;
    case 2: launch_pv_lat<2>(a, st); break;
    default: launch_pv_lat<1>(a, st); break;
  }
  if (cudaGetLastError() != cudaSuccess) return 1;
  pv_finish_kernel<<<rows, kTile, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
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

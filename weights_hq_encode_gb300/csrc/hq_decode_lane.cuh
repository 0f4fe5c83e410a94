// hq_decode_lane.cuh -- the per-group decoding step shared by the decoder and
// the fused kernels (scores, attention, weight products).
//
// A block of 256 threads decodes one index group of 32 tiles; lane r of a
// tile handles symbols 16r .. 16r+15 (two 8-vectors).  The block finds where
// every lane's unary codes start by a block-wide popcount scan of the U-area
// (every one bit there ends a symbol: 16 per lane).  Each lane reads its
// remainders at their fixed position and its unary codes with
// count-leading-zeros, restores the stripped bits, regenerates the dither and
// returns e = v - u in the lattice domain (HyperQuant summary, Method 2-4 in
// reverse).  Every loop is bounded by the group's word count from the index,
// and a group that fails any check yields zeros and a false return value.
#pragma once
#include <cuda_runtime.h>

#include "hq_device.cuh"
#include "hq_internal.h"

namespace hq {

constexpr int kDecThreads = 256;

// Synchronisation of the 256 threads that decode one group: the whole block
// (BlockBar), or team t = threadIdx.x / 256 of a larger block on named
// barrier 1 + t (TeamBar), so that several teams decode different groups
// independently.
struct BlockBar {
  __device__ static int tid() { return threadIdx.x; }
  __device__ static void sync() { __syncthreads(); }
  __device__ static int sync_or(int p) { return __syncthreads_or(p); }
  __device__ static int sync_and(int p) { return __syncthreads_and(p); }
};
struct TeamBar {
  __device__ static int tid() { return threadIdx.x & (kDecThreads - 1); }
  __device__ static uint32_t id() { return 1u + (threadIdx.x / kDecThreads); }
  __device__ static void sync() {
    asm volatile("bar.sync %0, %1;" ::"r"(id()), "n"(kDecThreads) : "memory");
  }
  __device__ static int sync_or(int p) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(p), "r"(id()), "n"(kDecThreads)
        : "memory");
    return r;
  }
  __device__ static int sync_and(int p) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(p), "r"(id()), "n"(kDecThreads)
        : "memory");
    return r;
  }
};

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

// MSB-first place (0..7) of each set bit of a byte: nibble k - 1 of
// entry b is the place of b's k-th set bit.
struct NthBitInByte {
  uint32_t v[256];
  constexpr NthBitInByte() : v() {
    for (int b = 0; b < 256; ++b) {
      uint32_t t = 0u;
      int k = 0;
      for (int i = 7; i >= 0; --i)
        if ((b >> i) & 1) t |= (uint32_t)(7 - i) << (4 * k++);
      v[b] = t;
    }
  }
};
__device__ const NthBitInByte kNthBitInByte = NthBitInByte();

// MSB-first position (0..31) of the n-th (1-based, n <= popc(x)) set bit of
// x: the byte holding it from the population counts of x's top 8, 16 and 24
// bits, its place inside the byte from the table.
__device__ __forceinline__ int nth_set_bit_msb(uint32_t x, int n) {
  const int c1 = __popc(x >> 24), c2 = __popc(x >> 16), c3 = __popc(x >> 8);
  const int k = (n > c1 ? 1 : 0) + (n > c2 ? 1 : 0) + (n > c3 ? 1 : 0);   // c1 <= c2 <= c3
  const int before = n > c3 ? c3 : n > c2 ? c2 : n > c1 ? c1 : 0;
  const uint32_t byte = (x >> (24 - 8 * k)) & 0xFFu;
  const uint32_t t = __ldg(&kNthBitInByte.v[byte]);
  return 8 * k + (int)((t >> (4 * (n - before - 1))) & 7u);
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
// return value is false when the group is corrupt (e is then all zeros):
// uniform over the decoding threads, or, with DEFER, this lane's own verdict.
template <int LAT, int K, class P, class Bar, bool DEFER>
__device__ __forceinline__ bool decode_lane_p(const DecodeArgs &a, int64_t g, int nt,
                                              const uint32_t *W, P nwords, bool bad,
                                              float e[16], P *s_start,
                                              uint32_t (*s_warp)[kDecThreads / 32]) {
  const int tid = Bar::tid(), tl = tid >> 3, r = tid & 7, lane = tid & 31, warp = tid >> 5;
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
      Bar::sync();
      // lane i < 8 takes warp i's total: two warp reductions give the ones
      // before this warp and the window's total (at most 8192: no wrap)
      static_assert(kDecThreads / 32 == 8, "one warp total per lane 0..7");
      const uint32_t wt = lane < kDecThreads / 32 ? s_warp[par][lane] : 0u;
      const uint32_t before_w = __reduce_add_sync(0xffffffffu, lane < warp ? wt : 0u);
      const uint32_t total = __reduce_add_sync(0xffffffffu, wt);
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
  Bar::sync();
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
  if constexpr (DEFER) {
    // the caller combines the lanes' verdicts at its own next barrier
    const bool mine = bad || lbad;
    if (mine || !valid) {
#pragma unroll
      for (int i = 0; i < 16; ++i) e[i] = 0.0f;
    }
    return !mine;
  } else {
    const int any_bad = Bar::sync_or((bad || lbad) ? 1 : 0);
    if (any_bad || !valid) {
#pragma unroll
      for (int i = 0; i < 16; ++i) e[i] = 0.0f;
    }
    return !any_bad;
  }
}

// Dispatch on the group's size: 32-bit bit positions unless the group holds
// 2^31 bits or more.  Without DEFER the return value is the group's verdict
// (uniform over the decoding threads) and a corrupt group yields zeros in
// every lane; with DEFER each lane returns its own verdict and zeroes only
// its own values, and the caller must OR the verdicts over the group (at a
// barrier it takes anyway) and treat the whole group as zeros if any lane
// failed.
template <int LAT, int K, class Bar = BlockBar, bool DEFER = false>
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
    return decode_lane_p<LAT, K, uint32_t, Bar, DEFER>(a, g, nt, W, (uint32_t)nwords, bad, e,
                                                  reinterpret_cast<uint32_t *>(s_start64), s_warp);
  return decode_lane_p<LAT, K, uint64_t, Bar, DEFER>(a, g, nt, W, nwords, bad, e, s_start64,
                                                     s_warp);
}

}  // namespace hq

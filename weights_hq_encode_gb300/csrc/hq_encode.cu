// hq_encode.cu -- single-pass encoder of the HyperQuant tile codec.
//
// A block of 256 threads codes one index group of 32 tiles; the 8 lanes
// r = 0..7 of a tile hold coordinates 16r .. 16r+15 (two 8-vectors), so the
// 32-byte loads of a warp are contiguous.  Per tile (HyperQuant summary,
// Method 1-4): apply the segment's sign mask to the bf16 input, FWHT-128
// (stages 1-8 in registers, then a transposition through shared memory so
// that stages 16-64 run in registers too), scale by alpha/sqrt(128) and add
// the subtractive dither in one fused multiply-add (on fp32 pairs), snap each
// 8-vector to the nearest lattice point and fold it into Rice symbols.
// Bit lengths are scanned across the 8 lanes of a tile and the 32 tiles of
// the group; groups are chained by a decoupled look-back (Merrill & Garland
// 2016) with bounded waits.  The group's words are assembled in shared memory
// by all warps; then warps 1-7 exit, so that their slots go to the next
// block, while warp 0 alone waits for the predecessors' prefix and stores
// the words with coalesced 32-bit writes.
#include <cuda_runtime.h>

#include "hq_device.cuh"
#include "hq_internal.h"

namespace hq {

constexpr int kEncThreads = 256;                 // one group of 32 tiles
constexpr int kStageWords = 4096;                // 16 KiB of output per window
constexpr int kKmaxTemplated = 8;                // Rice k specialised at compile time
// Dense rotation (optional), as a [32 tiles x 128] x [128 x 128] product in
// shared memory: the group's tiles [32][132] in the staging window (unused
// until the transform; later reused for the result), and the segment's R
// streamed in chunks of 16 columns, [128][20] each, two in flight
// (asynchronous copies): rows 80 bytes apart put the 16 rows a warp reads
// per request in two bank-conflict-free halves.
constexpr int kRotStride = kTile + 4;
constexpr int kRotXFloats = kGroupTiles * kRotStride;               // the group's tiles, then R x
constexpr int kRotChunk = 16, kRotChunkStride = kRotChunk + 4;
constexpr int kRotChunkFloats = kTile * kRotChunkStride;
constexpr size_t kEncRotSmemBytes = (size_t)(2 * kRotChunkFloats) * 4;

// Columns 16 q .. 16 q + 15 of R (row-major, 16-byte aligned) into a chunk
// buffer, 16-byte asynchronous copies by all threads; one commit group.
__device__ __forceinline__ void rot_chunk_async(float *dst, const float *R, int q, int tid) {
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(dst);
  for (int idx = tid; idx < kTile * kRotChunk / 4; idx += kEncThreads) {
    const int row = idx >> 2, c4 = idx & 3;
    const uint32_t d = base + 4u * (uint32_t)(row * kRotChunkStride + 4 * c4);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d),
                 "l"(R + row * kTile + kRotChunk * q + 4 * c4)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

constexpr uint64_t kFlagAgg = 1ull << 62;        // look-back state: [63:62] flag
constexpr uint64_t kFlagPrefix = 2ull << 62;     //                  [61:0] words
constexpr uint64_t kFlagPoison = 3ull << 62;
constexpr uint64_t kValueMask = (1ull << 62) - 1;

// The look-back state word packs a flag and a value into one 64-bit word
// that is written and read whole; nothing else is published through it, so
// relaxed GPU-scope accesses are enough (and polls do not order each other).
__device__ __forceinline__ void st_state(uint64_t *p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_state(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Decoupled look-back, split in two so that a block publishes its own total
// as early as possible and waits for its predecessors as late as possible.
__device__ __forceinline__ void publish_total(uint64_t *state, uint32_t blk, uint64_t agg) {
  st_state(state + blk, (blk == 0 ? kFlagPrefix : kFlagAgg) | agg);
}

// Exclusive prefix (in words) of block `blk`, whose own total is `agg`, read
// by one full warp.  Each poll loads 32 * kPer predecessors (lane l holds
// distances kPer*l+1 .. kPer*l+kPer), finds the nearest one whose inclusive prefix is known and
// sums the totals up to it; when a closer predecessor has published nothing
// yet the poll is repeated, and when no prefix is in the window the next
// window is read (kPer = 1 measured fastest).  Every wait is bounded by `spins` polls; a block that runs out, or
// meets a poisoned predecessor, poisons itself and returns false.  Lane 0
// publishes the block's own prefix and returns it.
__device__ bool lookback_warp(uint64_t *state, uint32_t blk, uint64_t agg, uint32_t spins,
                              uint64_t *excl_out) {
  constexpr int kPer = 1;
  const int lane = threadIdx.x & 31;
  uint64_t excl = 0;
  bool ok = true;
  int64_t p = (int64_t)blk - 1;                       // nearest predecessor not yet summed
  uint32_t n = 0;
  while (p >= 0) {
    uint64_t v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int64_t q = p - (int64_t)(kPer * lane + i);
      v[i] = q >= 0 ? ld_state(state + q) : kFlagPrefix;   // before block 0: prefix 0
    }
    // first prefix and first unpublished/poisoned entry of this lane, in distance order
    int first_p = kPer, first_bad = kPer;
    bool poison = false;
#pragma unroll
    for (int i = kPer - 1; i >= 0; --i) {
      const uint64_t f = v[i] & ~kValueMask;
      if (f == kFlagPrefix) first_p = i;
      if (f == 0 || f == kFlagPoison) first_bad = i;
      if (f == kFlagPoison) poison = true;
    }
    const uint32_t has_p = __ballot_sync(0xffffffffu, first_p < kPer);
    const int pl = has_p ? __ffs(has_p) - 1 : 32;             // lane of the nearest prefix
    // a gap (unpublished or poisoned) closer than the nearest prefix blocks progress
    const bool gap = (lane < pl && first_bad < kPer) || (lane == pl && first_bad < first_p);
    const uint32_t gaps = __ballot_sync(0xffffffffu, gap);
    if (gaps) {
      if (__ballot_sync(0xffffffffu, gap && poison)) { ok = false; break; }
      if (++n > spins) { ok = false; break; }
      __nanosleep(n < 64 ? 32 : 256);
      continue;
    }
    uint64_t sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane < pl || (lane == pl && i <= first_p)) sum += v[i] & kValueMask;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
    excl += sum;
    if (has_p) break;
    p -= 32 * kPer;
  }
  if (lane == 0) {
    st_state(state + blk, ok ? (kFlagPrefix | ((excl + agg) & kValueMask)) : kFlagPoison);
    *excl_out = excl;
  }
  return ok;
}

// MSB-first bit writer into the shared-memory window [lo, lo + kStageWords)
// of group words.  Whole words are OR-ed in (the first and last word of a
// writer's range may be shared with neighbouring lanes).
struct BitOut {
  uint32_t *stage;
  int64_t lo;
  int64_t w;       // word receiving the next completed 32 bits
  uint64_t acc;    // pending bits, right-aligned
  int n;           // number of pending bits (< 32 between calls)

  __device__ void begin(uint32_t *sm, int64_t window_lo, int64_t bitpos) {
    stage = sm;
    lo = window_lo;
    w = bitpos >> 5;
    n = (int)(bitpos & 31);
    acc = 0;
  }
  __device__ void emit(int64_t wi, uint32_t word) {
    if (word != 0u && wi >= lo && wi < lo + kStageWords) atomicOr(stage + (wi - lo), word);
  }
  // nb (0..32) bits, right-aligned in val with zeros above.
  __device__ void put(uint32_t val, int nb) {
    acc = (acc << nb) | val;
    n += nb;
    if (n >= 32) {
      n -= 32;
      emit(w++, (uint32_t)(acc >> n));
    }
  }
  __device__ void zeros(uint32_t count) {
    while (count >= 32u) { put(0u, 32); count -= 32u; }
    put(0u, (int)count);
  }
  __device__ void finish() {
    if (n > 0) emit(w, (uint32_t)(acc << (32 - n)));
  }
};

// OR nb (1..32) bits, right-aligned in v, into the shared-memory window at
// bit position bp (MSB-first, window-relative); they touch at most two words.
__device__ __forceinline__ void or_bits32(uint32_t *stage, uint32_t bp, uint32_t v, uint32_t nb) {
  const uint32_t t = v << (32u - nb);            // left-aligned
  const uint32_t o = bp & 31u;
  const uint32_t hi = t >> o, lo = shl_clamp(t, 32u - o);
  if (hi != 0u) atomicOr(stage + (bp >> 5), hi);
  if (lo != 0u) atomicOr(stage + (bp >> 5) + 1, lo);
}

// Kept remainder bits of one 8-group of symbols, MSB-first, right-aligned
// (rbits8<LAT>(K) bits, at most 64).
template <int LAT, int K>
__device__ __forceinline__ uint64_t r_bits_of(const uint32_t s[8]) {
  uint64_t acc = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int lowb = stripped_low_bits<LAT>(c, K);
    const int nb = K - lowb;
    if (nb > 0) acc = (acc << nb) | (uint64_t)((s[c] >> lowb) & ((1u << nb) - 1u));
  }
  return acc;
}

// Unary codes of 8 symbols one by one (codes longer than 32 bits in total).
__device__ __noinline__ void put_unary_slow(BitOut *o, uint4 qa, uint4 qb) {
  const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
  for (int i = 0; i < 8; ++i) {
    o->zeros(q[i]);
    o->put(1u, 1);
  }
}

// Unary codes (q zeros then a one) of one 8-group.
template <int K>
__device__ __forceinline__ void put_unary8(BitOut &o, const uint32_t s[8], int kk) {
  const int k = K >= 0 ? K : kk;
  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = s[i] >> k;
  // terminator positions (LSB-first) in one word when the 8 codes fit in 32 bits
  uint32_t T = q[0], pat = bit_at(q[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    T = T + 1u + q[i];
    pat |= bit_at(T);
  }
  const uint32_t L = T + 1u;
  if (L <= 32u) {
    o.put(__brev(pat) >> (32u - L), (int)L);
  } else if (L <= 64u) {
    // the same positions in a 64-bit pattern (bit_at returns 0 past 31)
    uint32_t lo = 0, hi = 0, P = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      P += q[i];
      lo |= bit_at(P);
      hi |= bit_at(P - 32u);
      P += 1u;
    }
    const uint64_t msb_first = ((uint64_t)__brev(lo) << 32 | __brev(hi)) >> (64u - L);
    if (L > 32u) o.put((uint32_t)(msb_first >> 32), (int)L - 32);
    o.put((uint32_t)msb_first, 32);
  } else {
    BitOut tmp = o;               // only the copy's address escapes: o stays in registers
    put_unary_slow(&tmp, make_uint4(q[0], q[1], q[2], q[3]), make_uint4(q[4], q[5], q[6], q[7]));
    o = tmp;
  }
}

// ROT: the dense-rotation variant (an instance of its own, 4 blocks per SM
// with the registers of its 4 x 4 product tile; runtime k only).
template <int LAT, int K, bool ROT>
__global__ void __launch_bounds__(kEncThreads, ROT ? 4 : 6)
encode_kernel(EncodeArgs a) {
  // staging window of the group's words; before that, the tile transposes of the transform
  __shared__ __align__(16) uint32_t s_stage[kStageWords > kGroupTiles * kTrTile ? kStageWords : kGroupTiles * kTrTile];
  __shared__ uint32_t s_tile_u[kGroupTiles];
  __shared__ uint64_t s_tile_uoff[kGroupTiles];
  __shared__ uint64_t s_base, s_words;
  __shared__ uint32_t s_ticket, s_flags;
  __shared__ int s_ok;
  // (dense rotation) sign XOR words of the segment; lane r's two 16-byte
  // blocks sit at r and 8 + r, so the 8 lanes of a tile read 128 contiguous
  // bytes
  __shared__ uint4 s_signx[ROT ? kTile / 8 : 1];


  const int tid = threadIdx.x, lane = tid & 31, tl = tid >> 3, r = tid & 7;
  uint64_t *state = reinterpret_cast<uint64_t *>(a.ws) + 1;
  // This block's group comes from the workspace's ticket counter, not from
  // the launch index: a block holding ticket g knows that the blocks holding
  // tickets 0 .. g-1 are already running, so its look-back always makes
  // progress whatever order the hardware starts blocks in.  (A counter set
  // ahead by the caller leaves groups unprocessed, which the bounded waits
  // turn into HQ_ERR_TIMEOUT.)
  if (tid == 0) {
    s_ticket = atomicAdd(reinterpret_cast<unsigned int *>(a.ws), 1u);
    s_flags = 0u;
  }
  __syncthreads();
  const uint32_t g = s_ticket;
  if (g >= a.n_blocks) return;                   // only with a counter set ahead
  const int k = K >= 0 ? K : a.rice_k;
  const int64_t t0 = (int64_t)g * kGroupTiles;
  const int nt = (int)min((int64_t)kGroupTiles, a.n_tiles - t0);
  const int64_t t = t0 + tl;
  const bool valid = tl < nt;
  // the lane's 16 bf16 coordinates and (without the rotation) the 16 sign
  // bits of its tile's mask, loaded together
  uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
  uint32_t mw = 0u;
  if (valid) {
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + t * kTile + 16 * r);
    v0 = __ldg(src);
    v1 = __ldg(src + 1);
    if constexpr (!ROT)
      mw = __ldg(a.signs + 4 * div_by(t, a.tiles_per_segment, a.seg_shift) + (r >> 1)) >> (16 * (r & 1));
  }
  const int64_t seg0 = div_by(t0, a.tiles_per_segment, a.seg_shift);
  if constexpr (ROT) {                           // R's first chunk arrives while the tiles are staged
    extern __shared__ __align__(16) float s_dyn_r[];   // the group is in one segment
    rot_chunk_async(s_dyn_r, a.rot + seg0 * (int64_t)(kTile * kTile), 0, tid);
  }
  if constexpr (ROT) {                           // the rotation applies the signs after its product
    if (tid < kTile / 2) {
      const uint32_t mword = __ldg(a.signs + 4 * seg0 + (tid >> 4));
      // word tid = pair q = tid & 7 of lane r = tid >> 3
      reinterpret_cast<uint32_t *>(s_signx)[32 * ((tid & 7) >> 2) + 4 * (tid >> 3) + (tid & 3)] =
          (((mword >> (2 * (tid & 15))) & 3u) * 0x40008000u) & 0x80008000u;
    }
    __syncthreads();
  }

  // ---- optional dense rotation R x (before the sign mask)
  float x[16];
  if constexpr (ROT) {
    extern __shared__ __align__(16) float s_dyn[];   // two chunks of R: [128][20] each
    const float *Rg = a.rot + seg0 * (int64_t)(kTile * kTile);
    float *s_x = reinterpret_cast<float *>(s_stage);   // [32][132]: coordinate j of tile t at [t][j]
    static_assert(kRotXFloats <= (int)(sizeof(s_stage) / 4), "the tiles fit the staging window");
    {
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      float4 *dst = reinterpret_cast<float4 *>(s_x + tl * kRotStride + 16 * r);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        dst[c] = make_float4(__uint_as_float(w[2 * c] << 16), __uint_as_float(w[2 * c] & 0xFFFF0000u),
                             __uint_as_float(w[2 * c + 1] << 16),
                             __uint_as_float(w[2 * c + 1] & 0xFFFF0000u));
    }
    // thread (tg, oh, l16): tiles 4 tg .. 4 tg + 3 x outputs 64 oh + l16 + 16 c
    // (c = 0..3), each output one fma chain over j = 0..127 from +0
    const int tg = (tid >> 4) & 7, ob = 64 * (tid >> 7) + (tid & 15);
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[u][c] = 0.0f;
#pragma unroll 1
    for (int q = 0; q < kTile / kRotChunk; ++q) {
      // chunk q has landed (chunk q + 1 is issued once every thread is past
      // chunk q - 1, whose buffer it reuses)
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();
      if (q + 1 < kTile / kRotChunk) rot_chunk_async(s_dyn + ((q + 1) & 1) * kRotChunkFloats, Rg, q + 1, tid);
      const float *s_r = s_dyn + (q & 1) * kRotChunkFloats;   // [128][20]: R[i][16 q + jj] at [i][jj]
#pragma unroll
      for (int jj = 0; jj < kRotChunk; jj += 4) {
        const int j = kRotChunk * q + jj;
        float4 xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          xv[u] = *reinterpret_cast<const float4 *>(s_x + (4 * tg + u) * kRotStride + j);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 rv = *reinterpret_cast<const float4 *>(s_r + (ob + 16 * c) * kRotChunkStride + jj);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[u][c] = __fmaf_rn(rv.x, xv[u].x, acc[u][c]);
            acc[u][c] = __fmaf_rn(rv.y, xv[u].y, acc[u][c]);
            acc[u][c] = __fmaf_rn(rv.z, xv[u].z, acc[u][c]);
            acc[u][c] = __fmaf_rn(rv.w, xv[u].w, acc[u][c]);
          }
        }
      }
    }
    __syncthreads();                             // the tile area becomes the result area
    float *s_z = s_x;                            // [32][132]
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) s_z[(4 * tg + u) * kRotStride + ob + 16 * c] = acc[u][c];
    __syncthreads();
    float z[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 q = *reinterpret_cast<const float4 *>(s_z + tl * kRotStride + 16 * r + 4 * c);
      z[4 * c] = q.x;
      z[4 * c + 1] = q.y;
      z[4 * c + 2] = q.z;
      z[4 * c + 3] = q.w;
    }
    __syncthreads();                             // every row is read before the transposes reuse the window
    const uint4 s0 = s_signx[r], s1 = s_signx[8 + r];
    const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {                // bf16-pair sign bits 15 / 31 -> fp32 bit 31
      x[2 * q] = __uint_as_float(__float_as_uint(z[2 * q]) ^ (sw[q] << 16));
      x[2 * q + 1] = __uint_as_float(__float_as_uint(z[2 * q + 1]) ^ (sw[q] & 0x80000000u));
    }
  } else if (valid) {
    // sign bits of coordinates 2q, 2q+1 moved to bit 15 / bit 31 of a bf16 pair
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t ww = w[q] ^ ((((mw >> (2 * q)) & 3u) * 0x40008000u) & 0x80008000u);
      x[2 * q] = __uint_as_float(ww << 16);
      x[2 * q + 1] = __uint_as_float(ww & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.0f;
  }
  // the staging window holds the tile transposes of the transform until the
  // group layout is known (it is cleared after the next block barrier)
  fwht128_t8(x, reinterpret_cast<float *>(s_stage) + tl * kTrTile, r);

  // ---- scale + dither (one rounding), range rule for the whole tile
  const uint64_t gt = a.tile_base + (uint64_t)t;
  bool bad = false;
  {
    float u[16];
    if (a.dither) {
      dither8<LAT>(a.keys, gt, (uint32_t)(2 * r), u);
      dither8<LAT>(a.keys, gt, (uint32_t)(2 * r + 1), u + 8);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] = 0.0f;
    }
    const uint64_t S2 = pk2(a.s_enc, a.s_enc);
#pragma unroll
    for (int i = 0; i < 8; ++i) upk2(fma2(pk2(x[i], x[8 + i]), S2, pk2(u[i], u[8 + i])), x[i], x[8 + i]);
    // range rule: a sum of magnitudes rounds to at least its largest term, so
    // a sum within the limit clears all 16 values (NaN and overflow fail it
    // and take the value-by-value test)
    float sa[4] = {fabsf(x[0]), fabsf(x[1]), fabsf(x[2]), fabsf(x[3])};
#pragma unroll
    for (int i = 4; i < 16; ++i) sa[i & 3] = __fadd_rn(sa[i & 3], fabsf(x[i]));
    if (!(__fadd_rn(__fadd_rn(sa[0], sa[1]), __fadd_rn(sa[2], sa[3])) <= kRangeLimit)) {
#pragma unroll
      for (int i = 0; i < 16; ++i) bad |= !(fabsf(x[i]) <= kRangeLimit);
    }
  }
  const uint32_t bal = __ballot_sync(0xffffffffu, valid && bad);
  if ((bal >> (lane & 24)) & 0xFFu) {            // some lane of this tile is out of range
    if (r == 0) atomicOr(&s_flags, (uint32_t)HQ_ERR_RANGE);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      float u[8];
      if (a.dither) {
        dither8<LAT>(a.keys, gt, (uint32_t)(2 * r + jj), u);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) u[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) x[8 * jj + i] = __fmaf_rn(0.0f, a.s_enc, u[i]);
    }
  }

  // ---- nearest point, fold, unary lengths
  uint32_t sym[16];
  if constexpr (LAT == 8) {
    quantize_fold16_e8(x, sym);
  } else {
    quantize_fold8<LAT>(x, sym);
    quantize_fold8<LAT>(x + 8, sym + 8);
  }
  uint32_t ubits = 0;
  if (valid) {
#pragma unroll
    for (int i = 0; i < 16; ++i) ubits += (sym[i] >> k) + 1u;
  }
  // prefix over the 8 lanes of the tile
  uint32_t incl = ubits;
#pragma unroll
  for (int d = 1; d < 8; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d, 8);
    if (r >= d) incl += o;
  }
  const uint32_t u_in_tile = incl - ubits;
  if (r == 7) s_tile_u[tl] = incl;
  __syncthreads();
  // the transposes are done: clear the staging window for the bit assembly
#pragma unroll
  for (int i = tid; i < kStageWords / 4; i += kEncThreads)
    reinterpret_cast<uint4 *>(s_stage)[i] = make_uint4(0u, 0u, 0u, 0u);

  // ---- group layout (warp 0): tile offsets, group total, published at once
  const uint64_t R = (uint64_t)(K >= 0 ? tile_rbits<LAT>(K) : a.rbits);
  if (tid < 32) {
    const uint64_t tu = s_tile_u[tid];
    uint64_t ui = tu;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t o = __shfl_up_sync(0xffffffffu, ui, d);
      if (lane >= d) ui += o;
    }
    s_tile_uoff[tid] = ui - tu;
    const uint64_t gbits = (uint64_t)nt * R + __shfl_sync(0xffffffffu, ui, 31);
    const uint64_t words = (gbits + 31) >> 5;
    if (tid == 0) {
      s_words = words;
      publish_total(state, g, words);
      if (a.payload_bits != nullptr) atomicAdd(a.payload_bits, (unsigned long long)gbits);
    }
  }
  __syncthreads();
  const uint64_t gwords = s_words;
  const int rb8 = K >= 0 ? rbits8<LAT>(K) : (int)(R / 16);
  const int64_t r_pos = (int64_t)tl * (int64_t)R + (int64_t)r * 2 * rb8;
  const int64_t u_pos = (int64_t)nt * (int64_t)R + (int64_t)s_tile_uoff[tl] + u_in_tile;
  const bool one_window = gwords <= (uint64_t)kStageWords;

  // ---- groups larger than the staging window: warp 0 waits for the
  // predecessors first, then every window is assembled and copied out
  if (!one_window && tid < 32) {
    uint64_t excl = 0;
    const bool ok = lookback_warp(state, g, gwords, a.spins, &excl);
    if (tid == 0) {
      s_ok = ok ? 1 : 0;
      s_base = excl;
      if (!ok) {
        atomicOr(a.status, (uint32_t)HQ_ERR_TIMEOUT);
      } else {
        if (a.offsets != nullptr) {
          a.offsets[g] = excl;
          if ((int64_t)g == a.n_groups - 1) a.offsets[a.n_groups] = excl + gwords;
        }
        if (excl + gwords > a.cap_words) atomicOr(a.status, (uint32_t)HQ_ERR_CAPACITY);
        if (s_flags) atomicOr(a.status, s_flags);
      }
    }
  }
  for (int64_t cb = 0; cb < (int64_t)gwords || cb == 0; cb += kStageWords) {
    if (!one_window) {                          // rare: groups beyond 16 KiB
      __syncthreads();
      for (int i = tid; i < kStageWords; i += kEncThreads) s_stage[i] = 0u;
      __syncthreads();
    }
    // unary bits of each 8-group of the lane (q zeros then a one per code)
    uint32_t la = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) la += (sym[i] >> k) + 1u;
    if (K >= 0 && 2 * rb8 <= 32 && one_window && valid && a.stream != nullptr && la <= 32u &&
        ubits - la <= 32u) {
      // common case: window-relative positions (below 2^17), the remainder
      // bits of the lane and each 8-group's unary codes in one 32-bit value
      if (rb8 > 0) {
        constexpr int KK = K >= 0 ? K : 0;
        constexpr int RB = 2 * rbits8<LAT>(KK) <= 32 ? rbits8<LAT>(KK) : 0;
        const uint32_t rv = ((uint32_t)r_bits_of<LAT, KK>(sym) << RB) |
                            (uint32_t)r_bits_of<LAT, KK>(sym + 8);
        or_bits32(s_stage, (uint32_t)r_pos, rv, (uint32_t)(2 * rb8));
      }
      uint32_t ua = 0u, ub = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ua = ((ua << (sym[i] >> k)) << 1) | 1u;
        ub = ((ub << (sym[8 + i] >> k)) << 1) | 1u;
      }
      or_bits32(s_stage, (uint32_t)u_pos, ua, la);
      or_bits32(s_stage, (uint32_t)u_pos + la, ub, ubits - la);
    } else if (valid && a.stream != nullptr) {
      BitOut o;
      if (rb8 > 0) {
        o.begin(s_stage, cb, r_pos);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          if (K >= 0) {
            const uint64_t rv = r_bits_of<LAT, (K >= 0 ? K : 0)>(sym + 8 * jj);
            if (rb8 > 32) o.put((uint32_t)(rv >> 32), rb8 - 32);
            o.put((uint32_t)rv & (rb8 >= 32 ? 0xFFFFFFFFu : ((1u << rb8) - 1u)),
                  rb8 > 32 ? 32 : rb8);
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int lowb = stripped_low_bits<LAT>(c, k);
              const int nb = k - lowb;
              if (nb > 0) o.put((sym[8 * jj + c] >> lowb) & ((1u << nb) - 1u), nb);
            }
          }
        }
        o.finish();
      }
      o.begin(s_stage, cb, u_pos);
      put_unary8<K>(o, sym, k);
      put_unary8<K>(o, sym + 8, k);
      o.finish();
    }
    __syncthreads();
    if (one_window) {
      // warps 1..7 are done and leave (their slots go to the next block);
      // warp 0 alone waits for the predecessors and copies the group out
      if (tid >= 32) return;
      uint64_t excl = 0;
      const bool ok = lookback_warp(state, g, gwords, a.spins, &excl);
      excl = __shfl_sync(0xffffffffu, excl, 0);
      if (tid == 0) {
        if (!ok) {
          atomicOr(a.status, (uint32_t)HQ_ERR_TIMEOUT);
        } else {
          if (a.offsets != nullptr) {
            a.offsets[g] = excl;
            if ((int64_t)g == a.n_groups - 1) a.offsets[a.n_groups] = excl + gwords;
          }
          if (excl + gwords > a.cap_words) atomicOr(a.status, (uint32_t)HQ_ERR_CAPACITY);
          if (s_flags) atomicOr(a.status, s_flags);
        }
      }
      if (!ok || a.stream == nullptr) return;
      for (int64_t i = tid; i < (int64_t)gwords; i += 32) {
        const uint64_t gw = excl + (uint64_t)i;
        if (gw < a.cap_words) a.stream[gw] = s_stage[i];
      }
      return;
    }
    if (!s_ok || a.stream == nullptr) return;
    const uint64_t base = s_base;
    const int64_t nw = min((int64_t)kStageWords, (int64_t)gwords - cb);
    for (int i = tid; i < nw; i += kEncThreads) {
      const uint64_t gw = base + (uint64_t)(cb + i);
      if (gw < a.cap_words) a.stream[gw] = s_stage[i];
    }
    if (one_window) break;
  }
}

template <int LAT, int K, bool ROT = false>
static void launch_one(const EncodeArgs &a, cudaStream_t st) {
  const size_t dyn = ROT ? kEncRotSmemBytes : 0;
  if (dyn)
    cudaFuncSetAttribute(encode_kernel<LAT, K, ROT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)dyn);
  encode_kernel<LAT, K, ROT><<<dim3((unsigned)a.n_blocks), dim3(kEncThreads), dyn, st>>>(a);
}

template <int LAT>
static void launch_lat(const EncodeArgs &a, cudaStream_t st) {
  if (a.rot != nullptr) {                        // the rotation variant takes k at run time
    launch_one<LAT, -1, true>(a, st);
    return;
  }
  switch (a.rice_k) {
    case 0: launch_one<LAT, 0>(a, st); break;
    case 1: launch_one<LAT, 1>(a, st); break;
    case 2: launch_one<LAT, 2>(a, st); break;
    case 3: launch_one<LAT, 3>(a, st); break;
    case 4: launch_one<LAT, 4>(a, st); break;
    case 5: launch_one<LAT, 5>(a, st); break;
    case 6: launch_one<LAT, 6>(a, st); break;
    case 7: launch_one<LAT, 7>(a, st); break;
    case 8: launch_one<LAT, 8>(a, st); break;
    default: launch_one<LAT, -1>(a, st); break;
  }
}

int launch_encode(const EncodeArgs &a, int lattice, cudaStream_t st) {
  static_assert(kKmaxTemplated == 8, "dispatch covers k = 0..8");
  switch (lattice) {
    case 8: launch_lat<8>(a, st); break;
    case 4: launch_lat<4>(a, st); break;
    case 2: launch_lat<2>(a, st); break;
    default: launch_lat<1>(a, st); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int encode_tiles_per_block() { return kGroupTiles; }

}  // namespace hq

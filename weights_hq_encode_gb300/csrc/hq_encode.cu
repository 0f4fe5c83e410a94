// hq_encode.cu -- single-pass encoder of the HyperQuant tile codec.
//
// One thread per 128-wide tile, one warp per index group of 32 tiles, one
// block of 128 threads per 4 groups.  Per tile (HyperQuant summary, Method
// 1-4): load bf16, apply the segment's sign mask, FWHT-128 in registers, scale
// by alpha/sqrt(128) and add the subtractive dither in one fused multiply-add,
// snap every 8-vector to the nearest lattice point, fold to Rice symbols.
// Bit lengths are scanned within the warp (group layout), across the block,
// and across blocks by a decoupled look-back (Merrill & Garland 2016) whose
// waits are bounded; the block then assembles its words in shared memory and
// stores them with coalesced 32-bit writes.
#include <cuda_runtime.h>

#include "hq_device.cuh"
#include "hq_internal.h"

namespace hq {

constexpr int kEncThreads = 128;                 // tiles per block
constexpr int kEncGroups = kEncThreads / 32;     // groups per block
constexpr int kStageWords = 6144;                // 24 KiB output staging per pass

// Look-back state word: [63:62] flag, [61:0] inclusive/aggregate word count.
constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagPrefix = 2ull << 62;
constexpr uint64_t kFlagPoison = 3ull << 62;
constexpr uint64_t kValueMask = (1ull << 62) - 1;

__device__ __forceinline__ void st_release(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Exclusive prefix (in words) of block `blk`, whose own total is `agg`.
// Returns false when a wait ran out or a predecessor was poisoned.
__device__ bool lookback(uint64_t *state, uint32_t blk, uint64_t agg, uint32_t spins,
                         uint64_t *excl_out) {
  if (blk == 0) {
    st_release(state, kFlagPrefix | agg);
    *excl_out = 0;
    return true;
  }
  st_release(state + blk, kFlagAgg | agg);
  uint64_t excl = 0;
  int64_t p = (int64_t)blk - 1;
  while (p >= 0) {
    uint64_t s;
    uint32_t n = 0;
    for (;;) {
      s = ld_acquire(state + p);
      if (s >> 62) break;
      if (++n > spins) {
        st_release(state + blk, kFlagPoison);
        return false;
      }
      __nanosleep(n < 64 ? 32 : 256);
    }
    if ((s & ~kValueMask) == kFlagPoison) {
      st_release(state + blk, kFlagPoison);
      return false;
    }
    excl += s & kValueMask;
    if ((s & ~kValueMask) == kFlagPrefix) break;
    --p;
  }
  st_release(state + blk, kFlagPrefix | ((excl + agg) & kValueMask));
  *excl_out = excl;
  return true;
}

// Appends bits MSB-first into a shared-memory window of words [cb, cb + kStageWords).
struct BitSink {
  uint32_t *sm;
  int64_t cb;
  int64_t cw;
  uint32_t cur;
  __device__ void flush() {
    if (cur != 0u && cw >= cb && cw < cb + kStageWords) atomicOr(sm + (cw - cb), cur);
    cur = 0u;
  }
  __device__ void or_word(int64_t w, uint32_t bits) {
    if (w != cw) { flush(); cw = w; }
    cur |= bits;
  }
  // nb (1..31) bits of val at bit position pos.
  __device__ void put(int64_t pos, uint32_t val, int nb) {
    int64_t w = pos >> 5;
    int sh = (int)(pos & 31);
    if (sh + nb <= 32) {
      or_word(w, val << (32 - sh - nb));
    } else {
      int lo = sh + nb - 32;                  // bits that spill into word w + 1
      or_word(w, val >> lo);
      or_word(w + 1, val << (32 - lo));
    }
  }
  __device__ void one(int64_t pos) { or_word(pos >> 5, 0x80000000u >> (pos & 31)); }
};

template <int LAT>
__global__ void __launch_bounds__(kEncThreads)
encode_kernel(EncodeArgs a) {
  __shared__ uint32_t s_stage[kStageWords];
  __shared__ uint64_t s_group_words[kEncGroups];
  __shared__ uint64_t s_base;
  __shared__ uint32_t s_ticket;
  __shared__ int s_ok;
  __shared__ uint32_t s_flags;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t *state = reinterpret_cast<uint64_t *>(a.ws) + 1;
  if (threadIdx.x == 0) {
    s_ticket = atomicAdd(reinterpret_cast<unsigned int *>(a.ws), 1u);
    s_flags = 0u;
  }
  __syncthreads();
  const uint32_t blk = s_ticket;
  if (blk >= a.n_blocks) return;               // only with a pre-filled ticket

  const int64_t t = (int64_t)blk * kEncThreads + threadIdx.x;
  const bool valid = t < a.n_tiles;
  const int k = a.rice_k;
  uint32_t sym[128];
  uint64_t ubits = 0;

  if (valid) {
    // ---- load, sign, FWHT
    float x[128];
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + t * kTile);
    const uint32_t *mask = a.signs + 4 * (t / a.tiles_per_segment);
    uint32_t m[4] = {__ldg(mask), __ldg(mask + 1), __ldg(mask + 2), __ldg(mask + 3)};
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      uint4 v = __ldg(src + c);
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        int i = 8 * c + 2 * h;
        uint32_t lo = w[h] << 16, hi = w[h] & 0xFFFF0000u;
        lo ^= ((m[i >> 5] >> (i & 31)) & 1u) << 31;
        hi ^= ((m[(i + 1) >> 5] >> ((i + 1) & 31)) & 1u) << 31;
        x[i] = __uint_as_float(lo);
        x[i + 1] = __uint_as_float(hi);
      }
    }
    fwht128(x);
    // ---- scale + dither (one rounding), range rule
    const uint64_t gt = a.tile_base + (uint64_t)t;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float u[8];
      if (a.dither) dither8<LAT>(a.dither_seed, gt, (uint32_t)j, u);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float y = __fmaf_rn(x[8 * j + i], a.s_enc, a.dither ? u[i] : 0.0f);
        bad |= !(fabsf(y) <= kRangeLimit);
        x[8 * j + i] = y;
      }
    }
    if (bad) {
      atomicOr(&s_flags, (uint32_t)HQ_ERR_RANGE);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float u[8];
        if (a.dither) dither8<LAT>(a.dither_seed, gt, (uint32_t)j, u);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          x[8 * j + i] = __fmaf_rn(0.0f, a.s_enc, a.dither ? u[i] : 0.0f);
      }
    }
    // ---- nearest point, fold, unary lengths
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      uint32_t s8[8];
      quantize_fold8<LAT>(x + 8 * j, s8);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sym[8 * j + i] = s8[i];
        ubits += (uint64_t)(s8[i] >> k) + 1u;
      }
    }
  }

  // ---- group layout: warp scan of unary lengths
  const int64_t g = (int64_t)blk * kEncGroups + warp;
  const int64_t gt0 = g * kGroupTiles;
  const int nt = (int)max((int64_t)0, min((int64_t)kGroupTiles, a.n_tiles - gt0));
  const uint64_t R = (uint64_t)a.rbits;
  uint64_t incl = ubits;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint64_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  const uint64_t u_excl = incl - ubits;
  const uint64_t group_bits = (uint64_t)nt * R + __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) s_group_words[warp] = (group_bits + 31) >> 5;
  __syncthreads();

  // ---- block scan + look-back
  if (threadIdx.x == 0) {
    uint64_t agg = 0;
    for (int w = 0; w < kEncGroups; ++w) agg += s_group_words[w];
    uint64_t excl = 0;
    bool ok = lookback(state, blk, agg, a.spins, &excl);
    if (!ok) atomicOr(a.status, (uint32_t)HQ_ERR_TIMEOUT);
    s_base = excl;
    s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  if (!s_ok) return;
  const uint64_t base = s_base;
  uint64_t gprefix = 0;
  for (int w = 0; w < warp; ++w) gprefix += s_group_words[w];
  uint64_t block_words = 0;
  for (int w = 0; w < kEncGroups; ++w) block_words += s_group_words[w];

  // ---- index
  if (lane == 0 && nt > 0) {
    a.offsets[g] = base + gprefix;
    if (g == a.n_groups - 1) a.offsets[a.n_groups] = base + gprefix + s_group_words[warp];
  }
  if (threadIdx.x == 0) {
    if (s_flags) atomicOr(a.status, s_flags);
    if (base + block_words > a.cap_words) atomicOr(a.status, (uint32_t)HQ_ERR_CAPACITY);
  }
  if (a.stream == nullptr) return;

  // ---- assemble words in shared memory, one window of kStageWords at a time
  const int64_t r_pos = (int64_t)(gprefix * 32 + (uint64_t)lane * R);
  const int64_t u_pos0 = (int64_t)(gprefix * 32 + (uint64_t)nt * R + u_excl);
  for (int64_t cb = 0; cb < (int64_t)block_words; cb += kStageWords) {
    for (int i = threadIdx.x; i < kStageWords; i += kEncThreads) s_stage[i] = 0u;
    __syncthreads();
    const int64_t lo_bit = cb * 32, hi_bit = (cb + kStageWords) * 32;
    if (valid) {
      BitSink sink{s_stage, cb, -1, 0u};
      // R-section (skipped when it lies outside the window)
      if (r_pos < hi_bit && r_pos + (int64_t)R > lo_bit && R > 0) {
        int64_t pos = r_pos;
#pragma unroll
        for (int j = 0; j < 128; ++j) {
          int lowb = stripped_low_bits<LAT>(j & 7, k);
          int nb = k - lowb;
          if (nb > 0) {
            sink.put(pos, (sym[j] >> lowb) & ((1u << nb) - 1u), nb);
            pos += nb;
          }
        }
      }
      // U-section
      if (u_pos0 < hi_bit && u_pos0 + (int64_t)ubits > lo_bit) {
        int64_t pos = u_pos0;
#pragma unroll
        for (int j = 0; j < 128; ++j) {
          pos += (int64_t)(sym[j] >> k);
          if (pos >= lo_bit && pos < hi_bit) sink.one(pos);
          ++pos;
        }
      }
      sink.flush();
    }
    __syncthreads();
    const int64_t nw = min((int64_t)kStageWords, (int64_t)block_words - cb);
    for (int i = threadIdx.x; i < nw; i += kEncThreads) {
      uint64_t gw = base + (uint64_t)(cb + i);
      if (gw < a.cap_words) a.stream[gw] = s_stage[i];
    }
    __syncthreads();
  }
}

int launch_encode(const EncodeArgs &a, int lattice, cudaStream_t st) {
  dim3 grid((unsigned)a.n_blocks), block(kEncThreads);
  switch (lattice) {
    case 8: encode_kernel<8><<<grid, block, 0, st>>>(a); break;
    case 4: encode_kernel<4><<<grid, block, 0, st>>>(a); break;
    default: encode_kernel<1><<<grid, block, 0, st>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int encode_tiles_per_block() { return kEncThreads; }

}  // namespace hq

// hq_internal.h -- argument blocks shared by the host entry points and the
// kernels of the codec library (not part of the public C ABI).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/hq.h"

namespace hq {

// Philox4x32-10 round keys of the dither seed (round r uses key + r * Weyl),
// precomputed on the host so the kernels read them from the parameter bank.
struct PhiloxKeys {
  uint32_t k0[10];
  uint32_t k1[10];
};

struct EncodeArgs {
  const uint16_t *x;
  int64_t n_tiles;
  int64_t n_groups;
  uint32_t n_blocks;
  uint32_t *stream;         // nullptr: size query
  uint64_t cap_words;
  uint64_t *offsets;
  void *ws;                 // [0]: ticket counter (uint32), then uint64 state[n_blocks]
  uint32_t *status;
  const uint32_t *signs;
  int64_t tiles_per_segment;
  int seg_shift;            // log2(tiles_per_segment) when a power of two, else -1
  uint64_t tile_base;
  uint64_t dither_seed;
  PhiloxKeys keys;
  float s_enc;
  int rice_k;
  int rbits;
  int dither;
  uint32_t spins;
  unsigned long long *payload_bits;   // non-null: add each group's Rice bits here
  const float *rot;         // nullptr, or [n_segments][128][128] row-major rotations
};

struct DecodeArgs {
  const uint32_t *stream;
  uint64_t stream_words;
  const uint64_t *offsets;
  int64_t n_tiles;
  int64_t n_groups;
  void *out;
  int out_kind;             // HQ_OUT_BF16 / HQ_OUT_F32; -1: lattice-domain e = v - u (fp32)
  uint32_t *status;
  const uint32_t *signs;
  int64_t tiles_per_segment;
  int seg_shift;            // log2(tiles_per_segment) when a power of two, else -1
  uint64_t tile_base;
  uint64_t dither_seed;
  PhiloxKeys keys;
  float s_dec;
  int rice_k;
  int rbits;
  int dither;
  const float *rot;         // nullptr, or [n_segments][128][128] row-major rotations
};

// Segment (or head) of tile t: a shift when the divisor is a power of two.
__host__ __device__ __forceinline__ int64_t div_by(int64_t t, int64_t d, int shift) {
  return shift >= 0 ? (t >> shift) : t / d;
}
__host__ __device__ __forceinline__ int pow2_shift(int64_t d) {
  if (d <= 0 || (d & (d - 1)) != 0) return -1;
  int s = 0;
  while ((1ll << s) < d) ++s;
  return s;
}

int launch_encode(const EncodeArgs &a, int lattice, cudaStream_t st);
int encode_tiles_per_block();
int launch_decode(const DecodeArgs &a, int lattice, cudaStream_t st);

}  // namespace hq

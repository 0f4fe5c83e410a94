// hq_fused.h -- arguments of the kernels that consume compressed tiles
// without writing them out (attention scores, decode attention, products
// with coded weights), shared by their launchers and the C ABI.
#pragma once
#include "hq_internal.h"

namespace hq {

struct QkArgs {
  DecodeArgs dec;           // K stream
  int n_kv;
  int64_t n_tokens;
  const uint16_t *q;        // [B][Hq][128] bf16
  int B, Hq;
  float *qrot;              // [B][Hq][128] fp32 workspace: s_dec * H * D_h * q
  float *scores;            // [B][Hq][n_tokens]
};

// Decode attention: the K side is the scores pass (qk), the V side another
// stream; each chunk of tokens keeps its own softmax maximum and sum (stats)
// beside its partial sums of exp(z - max) e (partials).
constexpr int kPvRows = 64;           // query rows per contraction tile
constexpr int kPvMinGroupsPerChunk = 4;  // smallest chunk (groups of 32 tokens) the launch may
                                         // pick; the workspace holds its chunk count
struct AttnArgs {
  QkArgs qk;                // K stream, queries, rotated queries, scores -> probabilities
  DecodeArgs v;             // V stream
  float scale;              // softmax scale applied to the scores
  float *partials;          // [n_kv][chunks][rowtiles][kPvRows][128]
  float2 *stats;            // [n_kv][chunks][rowtiles][kPvRows]: (max z, sum exp(z - max))
  int chunks, rowtiles;
  int pv_chunk;             // groups per chunk (set by the launch)
  float *out;               // [B][Hq][128] fp32
};

// Product with a compressed weight matrix W [rows][cols] (row-major tiles):
// y[b][o] = sum_i What[o][i] x[b][i].
struct GemmArgs {
  DecodeArgs dec;           // W stream
  int64_t rows, cols;
  int64_t tpr;              // tiles per row = cols / 128
  int tpr_shift;            // log2(tpr) when a power of two, else -1
  const uint16_t *x;        // [B][cols] bf16
  int B;
  float *xrot;              // [B][cols] fp32: s_dec * H * D * x, per 128-column tile
  float *partial;           // [B][n_tiles] fp32: one tile's share of y
  float *y;                 // [B][rows] fp32
  int fold_rows = 0;        // set by the launcher: tpr divides 32, so a row's tiles lie in
                            // one group and the product kernel sums them itself
};

int launch_decode_qk(const QkArgs &a, int lattice, cudaStream_t st);
int launch_decode_attention(const AttnArgs &a, int k_lattice, int v_lattice, bool want_probs,
                            cudaStream_t st);
int launch_decode_gemm(const GemmArgs &a, int lattice, cudaStream_t st);

}  // namespace hq

// hq_api.cu -- host entry points of the C ABI declared in include/hq.h.
// Argument checking, launch geometry and workspace layout; all arithmetic of
// the codec runs in the kernels.
#include <cmath>
#include <cstring>

#include <cuda_runtime.h>

#include "hq_fused.h"

namespace {

using namespace hq;

constexpr uint32_t kDefaultSpins = 1u << 20;   // ~0.3 s of polling per predecessor

bool lattice_ok(int l) { return l == HQ_Z || l == HQ_A2 || l == HQ_D4 || l == HQ_E8; }

int rbits_of(int lattice, int k) {
  // kept remainder bits per tile: 128 k minus the membership-fixed low bits
  int per8 = 0;
  for (int c = 0; c < 8; ++c) {
    int strip = 0;
    if (lattice == HQ_E8) strip = (c == 0) ? 0 : (c == 7 ? (k < 2 ? k : 2) : (k < 1 ? k : 1));
    else if (lattice == HQ_D4) strip = ((c & 3) == 3) ? (k < 1 ? k : 1) : 0;
    else if (lattice == HQ_A2) strip = (c & 1) ? (k < 1 ? k : 1) : 0;
    per8 += k - strip;
  }
  return per8 * 16;
}

bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

bool params_ok(const hq_params *p) {
  if (!p || !lattice_ok(p->lattice)) return false;
  if (p->d_rot && (!aligned(p->d_rot, 16) || p->tiles_per_segment <= 0 ||
                   p->tiles_per_segment % HQ_GROUP_TILES != 0))
    return false;
  if (p->rice_k < 0 || p->rice_k > 15) return false;
  if (!(p->alpha > 0.0f) || !std::isfinite(p->alpha)) return false;
  if (p->dither != 0 && p->dither != 1) return false;
  if (!p->d_signs || p->tiles_per_segment <= 0) return false;
  return true;
}


// Scales of the orthonormal RHT in lattice units, formed in double and
// rounded once (alpha / sqrt(128) forward, 1 / (alpha sqrt(128)) back).
float enc_scale(float alpha) { return (float)((double)alpha / std::sqrt(128.0)); }
float dec_scale(float alpha) { return (float)(1.0 / ((double)alpha * std::sqrt(128.0))); }

uint32_t host_philox_word_mul_hi(uint32_t a, uint32_t b) {
  return (uint32_t)(((uint64_t)a * b) >> 32);
}

PhiloxKeys round_keys(uint64_t seed) {
  PhiloxKeys k;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = k0;
    k.k1[r] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return k;
}

DecodeArgs make_decode_args(const hq_params *p, const uint32_t *stream, uint64_t stream_words,
                            const uint64_t *offsets, int64_t n_tiles, uint32_t *status) {
  DecodeArgs a;
  std::memset(&a, 0, sizeof a);
  a.stream = stream;
  a.stream_words = stream_words;
  a.offsets = offsets;
  a.n_tiles = n_tiles;
  a.n_groups = (n_tiles + HQ_GROUP_TILES - 1) / HQ_GROUP_TILES;
  a.status = status;
  a.signs = p->d_signs;
  a.tiles_per_segment = p->tiles_per_segment;
  a.seg_shift = pow2_shift(p->tiles_per_segment);
  a.tile_base = p->tile_base;
  a.dither_seed = p->dither_seed;
  a.keys = round_keys(p->dither_seed);
  a.s_dec = dec_scale(p->alpha);
  a.rice_k = p->rice_k;
  a.rbits = rbits_of(p->lattice, p->rice_k);
  a.dither = p->dither;
  a.rot = p->d_rot;
  return a;
}

}  // namespace

extern "C" {

int64_t hq_num_groups(int64_t n_tiles) {
  return n_tiles <= 0 ? 0 : (n_tiles + HQ_GROUP_TILES - 1) / HQ_GROUP_TILES;
}

size_t hq_encode_workspace_bytes(int64_t n_tiles) {
  int64_t tpb = hq::encode_tiles_per_block();
  int64_t blocks = n_tiles <= 0 ? 0 : (n_tiles + tpb - 1) / tpb;
  return 8 + 8 * (size_t)blocks;
}

namespace {

// hq_encode, plus the optional payload counter of hq_payload_bits.
int encode_impl(const hq_params *p, const uint16_t *d_x, int64_t n_tiles, uint32_t *d_stream,
                uint64_t cap_words, uint64_t *d_offsets, void *d_ws, size_t ws_bytes,
                uint32_t *d_status, cudaStream_t st, unsigned long long *d_bits) {
  if (n_tiles == 0) {
    if (d_offsets == nullptr) return HQ_OK;
    return cudaMemsetAsync(d_offsets, 0, sizeof(uint64_t), st) == cudaSuccess ? HQ_OK
                                                                             : HQ_ERR_CUDA;
  }
  if (!d_x || !aligned(d_x, 16) || !d_ws || !aligned(d_ws, 8) ||
      ws_bytes < hq_encode_workspace_bytes(n_tiles) || (d_offsets && !aligned(d_offsets, 8)))
    return HQ_ERR_INVALID;
  EncodeArgs a;
  std::memset(&a, 0, sizeof a);
  a.x = d_x;
  a.n_tiles = n_tiles;
  a.n_groups = hq_num_groups(n_tiles);
  int64_t tpb = hq::encode_tiles_per_block();
  int64_t blocks = (n_tiles + tpb - 1) / tpb;
  if (blocks > 0x7FFFFFFF) return HQ_ERR_INVALID;
  a.n_blocks = (uint32_t)blocks;
  a.stream = d_stream;
  // a size query reports the capacity it would need; a payload count does not
  a.cap_words = d_stream ? cap_words : (d_bits ? UINT64_MAX : 0);
  a.offsets = d_offsets;
  a.ws = d_ws;
  a.status = d_status;
  a.signs = p->d_signs;
  a.tiles_per_segment = p->tiles_per_segment;
  a.seg_shift = pow2_shift(p->tiles_per_segment);
  a.tile_base = p->tile_base;
  a.dither_seed = p->dither_seed;
  a.keys = round_keys(p->dither_seed);
  a.s_enc = enc_scale(p->alpha);
  a.rice_k = p->rice_k;
  a.rbits = rbits_of(p->lattice, p->rice_k);
  a.dither = p->dither;
  a.spins = p->lookback_spins ? p->lookback_spins : kDefaultSpins;
  a.payload_bits = d_bits;
  a.rot = p->d_rot;
  if (!(p->flags & HQ_FLAG_WORKSPACE_READY)) {
    if (cudaMemsetAsync(d_ws, 0, hq_encode_workspace_bytes(n_tiles), st) != cudaSuccess)
      return HQ_ERR_CUDA;
  }
  return hq::launch_encode(a, p->lattice, st) == 0 ? HQ_OK : HQ_ERR_CUDA;
}

}  // namespace

int hq_encode(const hq_params *p, const uint16_t *d_x, int64_t n_tiles, uint32_t *d_stream,
              uint64_t cap_words, uint64_t *d_offsets, void *d_ws, size_t ws_bytes,
              uint32_t *d_status, hq_stream_t stream) {
  if (!params_ok(p) || n_tiles < 0 || !d_offsets || !d_status) return HQ_ERR_INVALID;
  return encode_impl(p, d_x, n_tiles, d_stream, cap_words, d_offsets, d_ws, ws_bytes, d_status,
                     reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int hq_payload_bits(const hq_params *p, const uint16_t *d_x, int64_t n_tiles, uint64_t *d_bits,
                    void *d_ws, size_t ws_bytes, uint32_t *d_status, hq_stream_t stream) {
  if (!params_ok(p) || n_tiles < 0 || !d_bits || !aligned(d_bits, 8) || !d_status)
    return HQ_ERR_INVALID;
  return encode_impl(p, d_x, n_tiles, nullptr, 0, nullptr, d_ws, ws_bytes, d_status,
                     reinterpret_cast<cudaStream_t>(stream),
                     reinterpret_cast<unsigned long long *>(d_bits));
}

namespace {

// One rate evaluation of hq_calibrate: payload bits per element of the call's
// tiles at (alpha, k), read back synchronously.
int calib_rate(const hq_params &base, float alpha, int k, const uint16_t *d_x, int64_t n_tiles,
               void *d_ws, size_t ws_bytes, uint64_t *d_bits, uint32_t *d_status,
               cudaStream_t st, double *rate) {
  hq_params q = base;
  q.alpha = alpha;
  q.rice_k = k;
  q.flags &= ~HQ_FLAG_WORKSPACE_READY;
  if (cudaMemsetAsync(d_bits, 0, sizeof(uint64_t), st) != cudaSuccess ||
      cudaMemsetAsync(d_status, 0, sizeof(uint32_t), st) != cudaSuccess)
    return HQ_ERR_CUDA;
  int rc = hq_payload_bits(&q, d_x, n_tiles, d_bits, d_ws, ws_bytes, d_status,
                           reinterpret_cast<hq_stream_t>(st));
  if (rc != HQ_OK) return rc;
  uint64_t bits = 0;
  uint32_t status = 0;
  if (cudaMemcpyAsync(&bits, d_bits, sizeof bits, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(&status, d_status, sizeof status, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return HQ_ERR_CUDA;
  if (status & HQ_ERR_TIMEOUT) return HQ_ERR_CUDA;
  *rate = (double)bits / ((double)n_tiles * HQ_TILE);
  return HQ_OK;
}

}  // namespace

int hq_calibrate(const hq_params *p, const uint16_t *d_x, int64_t n_tiles, double target_bps,
                 double tol, int k_min, int k_max, void *d_ws, size_t ws_bytes,
                 uint64_t *d_bits, uint32_t *d_status, hq_stream_t stream,
                 hq_calibration *out) {
  if (!p || !out || n_tiles <= 0 || !(target_bps > 0.0) || !(tol > 0.0) || k_min < 0 ||
      k_max > 15 || k_min > k_max || !d_bits || !d_status)
    return HQ_ERR_INVALID;
  hq_params base = *p;
  base.alpha = 1.0f;
  base.rice_k = k_min;
  if (!params_ok(&base)) return HQ_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  std::memset(out, 0, sizeof *out);
  bool have = false;
  for (int k = k_min; k <= k_max; ++k) {
    // bisection on log2(alpha) over [-14, 18]; a k whose rate at the smallest
    // alpha is already above the target cannot reach it
    double lo = -14.0, hi = 18.0, r = 0.0;
    int rc = calib_rate(base, (float)std::pow(2.0, lo), k, d_x, n_tiles, d_ws, ws_bytes, d_bits,
                        d_status, st, &r);
    if (rc != HQ_OK) return rc;
    ++out->evaluations;
    if (r > target_bps - tol / 2) continue;
    bool have_best = false;
    double best_mid = 0.0, best_r = 0.0;
    for (int it = 0; it < 60; ++it) {
      const double mid = 0.5 * (lo + hi);
      rc = calib_rate(base, (float)std::pow(2.0, mid), k, d_x, n_tiles, d_ws, ws_bytes, d_bits,
                      d_status, st, &r);
      if (rc != HQ_OK) return rc;
      ++out->evaluations;
      if (!have_best || std::fabs(r - target_bps) < std::fabs(best_r - target_bps)) {
        have_best = true;
        best_mid = mid;
        best_r = r;
      }
      if (std::fabs(r - target_bps) <= tol) break;
      if (r < target_bps) lo = mid;
      else hi = mid;
    }
    const float alpha = (float)std::pow(2.0, best_mid);
    double bps = 0.0;
    rc = calib_rate(base, alpha, k, d_x, n_tiles, d_ws, ws_bytes, d_bits, d_status, st, &bps);
    if (rc != HQ_OK) return rc;
    ++out->evaluations;
    if (!(std::fabs(bps - target_bps) <= tol)) continue;
    // keep the largest alpha (least distortion); among equal alphas the smaller k
    if (!have || alpha > out->alpha) {
      have = true;
      out->alpha = alpha;
      out->rice_k = k;
      out->bps = bps;
    }
  }
  out->feasible = have ? 1 : 0;
  return HQ_OK;
}

int hq_decode(const hq_params *p, const uint32_t *d_stream, uint64_t stream_words,
              const uint64_t *d_offsets, int64_t n_tiles, void *d_out, int out_kind,
              uint32_t *d_status, hq_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!params_ok(p) || n_tiles < 0 || !d_status) return HQ_ERR_INVALID;
  if (out_kind != HQ_OUT_BF16 && out_kind != HQ_OUT_F32) return HQ_ERR_INVALID;
  if (n_tiles == 0) return HQ_OK;
  if (!d_stream || !d_offsets || !d_out || !aligned(d_out, 16) || !aligned(d_offsets, 8))
    return HQ_ERR_INVALID;
  DecodeArgs a = make_decode_args(p, d_stream, stream_words, d_offsets, n_tiles, d_status);
  a.out = d_out;
  a.out_kind = out_kind;
  return hq::launch_decode(a, p->lattice, st) == 0 ? HQ_OK : HQ_ERR_CUDA;
}

namespace {

// Attention workspace geometry: rotated queries, scores (probabilities),
// then the partial P . E rows of every (head, chunk, row tile).
struct AttnGeometry {
  int64_t chunks = 0, rowtiles = 0;
  size_t qrot = 0, scores = 0, partials = 0, stats = 0;
};

bool attn_geometry(int n_kv, int64_t n_tokens, int B, int Hq, AttnGeometry *g) {
  if (n_kv <= 0 || n_tokens <= 0 || B <= 0 || Hq <= 0 || Hq % n_kv != 0) return false;
  const int64_t rows = (int64_t)B * (Hq / n_kv);
  const int64_t groups = (n_tokens + HQ_GROUP_TILES - 1) / HQ_GROUP_TILES + 1;   // a head's groups
  // sized for the smallest chunk the launch may pick
  g->chunks = (groups + hq::kPvMinGroupsPerChunk - 1) / hq::kPvMinGroupsPerChunk;
  g->rowtiles = (rows + hq::kPvRows - 1) / hq::kPvRows;
  if (g->chunks > 0x7FFFFFFF || g->rowtiles > 65535 || n_kv > 65535) return false;
  // every region starts on a 256-byte boundary (the kernels use 16-byte vectors)
  auto round256 = [](size_t v) { return (v + 255) / 256 * 256; };
  g->qrot = round256((size_t)B * Hq * HQ_TILE * sizeof(float));
  g->scores = round256((size_t)B * Hq * (size_t)n_tokens * sizeof(float));
  g->partials = (size_t)n_kv * g->chunks * g->rowtiles * hq::kPvRows * HQ_TILE * sizeof(float);
  g->stats = (size_t)n_kv * g->chunks * g->rowtiles * hq::kPvRows * 2 * sizeof(float);
  return true;
}

}  // namespace

size_t hq_decode_attention_workspace_bytes(int n_kv_heads, int64_t n_tokens, int B, int Hq) {
  AttnGeometry g;
  if (!attn_geometry(n_kv_heads, n_tokens, B, Hq, &g)) return 0;
  return g.qrot + g.scores + g.partials + g.stats;
}

int hq_decode_attention(const hq_params *pk, const uint32_t *d_k_stream, uint64_t k_words,
                        const uint64_t *d_k_offsets, const hq_params *pv,
                        const uint32_t *d_v_stream, uint64_t v_words,
                        const uint64_t *d_v_offsets, int n_kv_heads, int64_t n_tokens,
                        const uint16_t *d_q, int B, int Hq, float scale, float *d_out,
                        float *d_probs, void *d_ws, size_t ws_bytes, uint32_t *d_status,
                        hq_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!params_ok(pk) || !params_ok(pv) || !d_status || !(scale == scale)) return HQ_ERR_INVALID;
  if (B == 0) return HQ_OK;
  AttnGeometry g;
  if (!attn_geometry(n_kv_heads, n_tokens, B, Hq, &g)) return HQ_ERR_INVALID;
  if (pk->tiles_per_segment % n_tokens != 0 || pv->tiles_per_segment % n_tokens != 0)
    return HQ_ERR_INVALID;
  if (!d_k_stream || !d_k_offsets || !d_v_stream || !d_v_offsets || !d_q || !d_out || !d_ws ||
      ws_bytes < g.qrot + g.scores + g.partials + g.stats || !aligned(d_ws, 16) ||
      !aligned(d_out, 16) ||
      !aligned(d_k_offsets, 8) || !aligned(d_v_offsets, 8) || (d_probs && !aligned(d_probs, 4)))
    return HQ_ERR_INVALID;
  char *ws = reinterpret_cast<char *>(d_ws);
  hq::AttnArgs a;
  const int64_t n_tiles = (int64_t)n_kv_heads * n_tokens;
  a.qk.dec = make_decode_args(pk, d_k_stream, k_words, d_k_offsets, n_tiles, d_status);
  a.qk.dec.out_kind = -1;
  a.qk.n_kv = n_kv_heads;
  a.qk.n_tokens = n_tokens;
  a.qk.q = d_q;
  a.qk.B = B;
  a.qk.Hq = Hq;
  a.qk.qrot = reinterpret_cast<float *>(ws);
  a.qk.scores = d_probs ? d_probs : reinterpret_cast<float *>(ws + g.qrot);
  a.v = make_decode_args(pv, d_v_stream, v_words, d_v_offsets, n_tiles, d_status);
  a.v.out_kind = -1;
  a.scale = scale;
  a.partials = reinterpret_cast<float *>(ws + g.qrot + g.scores);
  a.stats = reinterpret_cast<float2 *>(ws + g.qrot + g.scores + g.partials);
  a.chunks = (int)g.chunks;                     // the launch lowers it to its chunk size
  a.rowtiles = (int)g.rowtiles;
  a.out = d_out;
  return hq::launch_decode_attention(a, pk->lattice, pv->lattice, d_probs != nullptr, st) == 0
             ? HQ_OK
             : HQ_ERR_CUDA;
}

namespace {

bool gemm_sizes(int64_t rows, int64_t cols, int B, size_t *xrot, size_t *partial) {
  if (rows <= 0 || cols <= 0 || cols % HQ_TILE != 0 || B <= 0) return false;
  const int64_t n_tiles = rows * (cols / HQ_TILE);
  if (n_tiles / rows != cols / HQ_TILE || (int64_t)B * rows > ((int64_t)1 << 40)) return false;
  *xrot = ((size_t)B * cols * sizeof(float) + 255) / 256 * 256;
  *partial = (size_t)B * n_tiles * sizeof(float);
  return true;
}

}  // namespace

size_t hq_decode_gemm_workspace_bytes(int64_t rows, int64_t cols, int B) {
  size_t xr = 0, pa = 0;
  return gemm_sizes(rows, cols, B, &xr, &pa) ? xr + pa : 0;
}

int hq_decode_gemm(const hq_params *p, const uint32_t *d_w_stream, uint64_t w_words,
                   const uint64_t *d_w_offsets, int64_t rows, int64_t cols, const uint16_t *d_x,
                   int B, float *d_y, void *d_ws, size_t ws_bytes, uint32_t *d_status,
                   hq_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!params_ok(p) || !d_status) return HQ_ERR_INVALID;
  size_t xr = 0, pa = 0;
  if (!gemm_sizes(rows, cols, B, &xr, &pa)) return HQ_ERR_INVALID;
  const int64_t n_tiles = rows * (cols / HQ_TILE);
  if (n_tiles > p->tiles_per_segment) return HQ_ERR_INVALID;   // one sign segment
  if (!d_w_stream || !d_w_offsets || !d_x || !d_y || !d_ws || ws_bytes < xr + pa ||
      !aligned(d_ws, 16) || !aligned(d_w_offsets, 8))
    return HQ_ERR_INVALID;
  hq::GemmArgs a;
  a.dec = make_decode_args(p, d_w_stream, w_words, d_w_offsets, n_tiles, d_status);
  a.dec.out_kind = -1;
  a.rows = rows;
  a.cols = cols;
  a.tpr = cols / HQ_TILE;
  a.tpr_shift = pow2_shift(a.tpr);
  a.x = d_x;
  a.B = B;
  a.xrot = reinterpret_cast<float *>(d_ws);
  a.partial = reinterpret_cast<float *>(reinterpret_cast<char *>(d_ws) + xr);
  a.y = d_y;
  return hq::launch_decode_gemm(a, p->lattice, st) == 0 ? HQ_OK : HQ_ERR_CUDA;
}

size_t hq_decode_qk_workspace_bytes(int B, int Hq) {
  if (B <= 0 || Hq <= 0) return 0;
  return (size_t)B * (size_t)Hq * HQ_TILE * sizeof(float);
}

int hq_decode_qk(const hq_params *p, const uint32_t *d_k_stream, uint64_t stream_words,
                 const uint64_t *d_k_offsets, int n_kv_heads, int64_t n_tokens,
                 const uint16_t *d_q, int B, int Hq, float *d_scores, void *d_ws,
                 size_t ws_bytes, uint32_t *d_status, hq_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!params_ok(p) || !d_status || n_kv_heads <= 0 || n_tokens < 0 || B < 0 || Hq <= 0)
    return HQ_ERR_INVALID;
  if (Hq % n_kv_heads != 0) return HQ_ERR_INVALID;
  if (n_tokens == 0 || B == 0) return HQ_OK;
  if (p->tiles_per_segment % n_tokens != 0) return HQ_ERR_INVALID;
  if (!d_k_stream || !d_k_offsets || !d_q || !d_scores || !d_ws ||
      ws_bytes < hq_decode_qk_workspace_bytes(B, Hq) || !aligned(d_ws, 16) ||
      !aligned(d_k_offsets, 8))
    return HQ_ERR_INVALID;
  QkArgs a;
  a.dec = make_decode_args(p, d_k_stream, stream_words, d_k_offsets,
                           (int64_t)n_kv_heads * n_tokens, d_status);
  a.dec.out_kind = -1;
  a.n_kv = n_kv_heads;
  a.n_tokens = n_tokens;
  a.q = d_q;
  a.B = B;
  a.Hq = Hq;
  a.qrot = reinterpret_cast<float *>(d_ws);
  a.scores = d_scores;
  return hq::launch_decode_qk(a, p->lattice, st) == 0 ? HQ_OK : HQ_ERR_CUDA;
}

// Philox4x32-10 on the host (Salmon et al., SC'11), used for the sign masks.
void hq_make_signs(uint64_t seed, uint64_t segment, uint32_t out[4]) {
  uint32_t c0 = (uint32_t)segment, c1 = (uint32_t)(segment >> 32), c2 = 0u, c3 = 0x5349474Eu;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0 = host_philox_word_mul_hi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    uint32_t hi1 = host_philox_word_mul_hi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

void hq_make_layer_signs(uint64_t seed_d, uint64_t seed_s, uint64_t layer, uint32_t out[4]) {
  uint32_t d[4], sl[4];
  hq_make_signs(seed_d, 0, d);
  hq_make_signs(seed_s, layer, sl);
  for (int i = 0; i < 4; ++i) out[i] = d[i] ^ sl[i];
}

const char *hq_status_string(int status) {
  switch (status) {
    case HQ_OK: return "ok";
    case HQ_ERR_INVALID: return "invalid argument";
    case HQ_ERR_CUDA: return "CUDA launch failed";
    case HQ_ERR_CAPACITY: return "stream capacity exceeded";
    case HQ_ERR_CORRUPT: return "corrupt stream";
    case HQ_ERR_TIMEOUT: return "cross-block wait timed out";
    case HQ_ERR_RANGE: return "input out of range";
    default: return status < 0 ? "unknown status" : "several errors";
  }
}

}  // extern "C"

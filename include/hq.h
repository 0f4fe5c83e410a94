/*
 * hq.h -- C ABI of the GB300 (sm_103a) HyperQuant tile codec.
 *
 * The codec follows the HyperQuant technical summary, Method sections 1-4:
 *   1 "Per-tile randomized Hadamard transform": 128-wide tiles, RHT = H D x;
 *   2 "Lattice quantization": alpha scaling, nearest point of E8 (integer
 *     embedding 2E8 in Z^8), D4 or Z;
 *   3 "Bit stripping and Rice coding": membership-fixed bits removed, the
 *     remaining symbols Rice coded with parameter k;
 *   4 "Bias correction for the KV cache": per-layer +-1 sign rotation (folded
 *     into the per-segment sign masks) and subtractive dither
 *     U ~ Uniform(V(Lambda)), regenerated from a seed by the decoder.
 * and, for hq_decode_qk, the closing section's "fused decode + MMA" (attention
 * scores computed from compressed K without materialising K).
 *
 * Conventions for every entry point:
 *   - All pointers named d_* are device pointers (CUDA global memory); the
 *     caller allocates, owns and frees every buffer.  The library allocates
 *     nothing and keeps no state between calls, so calls on different
 *     streams are independent.  Every entry point is asynchronous except
 *     hq_calibrate, a host loop that reads each rate back.
 *   - The return value reports synchronous errors only: HQ_ERR_INVALID for a
 *     bad argument (nothing is launched), HQ_ERR_CUDA for a failed launch.
 *   - Data-dependent errors are OR-ed into *d_status (a device uint32 the
 *     caller zeroes beforehand and reads after its own synchronisation):
 *     HQ_ERR_CAPACITY, HQ_ERR_CORRUPT, HQ_ERR_TIMEOUT, HQ_ERR_RANGE.
 *   - bf16 data is passed as raw 16-bit patterns (uint16_t); fp32 as float.
 *   - The stream argument is a cudaStream_t (0 = legacy default stream).
 *
 * Stream format (one encode call):
 *   tiles are indexed in groups of HQ_GROUP_TILES = 32 consecutive tiles; each
 *   group starts on a 32-bit word boundary and holds
 *     R-area: for each tile, the kept remainder bits of its 128 Rice symbols
 *             (bits k-1..0 of each symbol, membership-fixed bits skipped);
 *     U-area: for each tile, for each symbol, q = s >> k zeros then a one;
 *     zero padding to the next word.
 *   Bit b of a group is bit 31 - (b % 32) of word b / 32 (MSB first).
 *   offsets[g] = word index of group g, offsets[n_groups] = total words.
 */
#ifndef HQ_H_
#define HQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *hq_stream_t;   /* same type as cudaStream_t */

/* Status bits (return values and *d_status). */
enum {
  HQ_OK = 0,
  HQ_ERR_INVALID = 1,   /* bad argument; nothing launched */
  HQ_ERR_CUDA = 2,      /* kernel launch or memset failed */
  HQ_ERR_CAPACITY = 4,  /* stream larger than cap_words: words past the cap
                           were not written; offsets are still complete */
  HQ_ERR_CORRUPT = 8,   /* a group failed a format check: its tiles decode to 0 */
  HQ_ERR_TIMEOUT = 16,  /* a bounded wait ran out (encode look-back, tensor-core completion) */
  HQ_ERR_RANGE = 32     /* non-finite input or |alpha * RHT(x)| > 2^20: the tile
                           was coded as an all-zero tile */
};

enum { HQ_Z = 1, HQ_A2 = 2, HQ_D4 = 4, HQ_E8 = 8 };   /* lattice = its dimension */
enum { HQ_OUT_BF16 = 0, HQ_OUT_F32 = 1 };

#define HQ_TILE 128
#define HQ_GROUP_TILES 32

/* Codec parameters, identical for the encode and decode of one stream.
 *   lattice            HQ_E8 (2E8 in Z^8), HQ_D4, HQ_A2 (hexagonal lattice,
 *                      codes (m, n) with m = n mod 2 for the point
 *                      (m/2, (sqrt 3/2) n)) or HQ_Z.
 *   rice_k             Rice parameter, 0..15.
 *   alpha              > 0: lattice units per unit of the orthonormal RHT
 *                      (H / sqrt(128)) output.
 *   dither             0 or 1 (subtractive dither, Method 4).
 *   dither_seed        Philox key of the dither.
 *   tile_base          global index of the call's first tile; the dither of
 *                      tile t of the call uses counter tile_base + t, so a
 *                      tensor split over several calls codes identically.
 *   d_signs            device [n_segments][4] uint32 sign masks (bit i of the
 *                      128-bit mask set = coordinate i negated before H), e.g.
 *                      hq_make_signs(seedD, 0) XOR hq_make_signs(seedS, layer).
 *   tiles_per_segment  > 0: tile t of the call uses mask t / tiles_per_segment.
 *   lookback_spins     0 = default; otherwise the bound on polls of one
 *                      predecessor in the encoder's cross-block scan, after
 *                      which HQ_ERR_TIMEOUT is raised.
 *   flags              bit 0 (HQ_FLAG_WORKSPACE_READY): the caller has zeroed
 *                      the encode workspace itself and hq_encode skips its
 *                      memset; the output is the same.  (Encoder blocks
 *                      always take their groups from the workspace's ticket
 *                      counter, one atomic per block, so that the cross-block
 *                      scan progresses whatever order blocks start in.)
 *   d_rot              NULL, or device [n_segments][128][128] fp32 row-major
 *                      per-layer dense rotations R (Method 3-4: a full
 *                      Haar-uniform QJL matrix instead of the +-1 diagonal):
 *                      tile t of segment s is coded as RHT(R_s x), each
 *                      (R x)_i one fused multiply-add chain over j = 0..127
 *                      from +0, and decoded with R_s^T applied after the
 *                      inverse transform (chain over i).  16-byte aligned;
 *                      tiles_per_segment must then be a multiple of 32. */
typedef struct hq_params {
  int32_t lattice;
  int32_t rice_k;
  float alpha;
  int32_t dither;
  uint64_t dither_seed;
  uint64_t tile_base;
  const uint32_t *d_signs;
  int64_t tiles_per_segment;
  uint32_t lookback_spins;
  uint32_t flags;
  const float *d_rot;
} hq_params;

#define HQ_FLAG_WORKSPACE_READY 1u

/* Number of index groups for n_tiles tiles: ceil(n_tiles / 32). */
int64_t hq_num_groups(int64_t n_tiles);

/* Bytes of device workspace hq_encode needs for n_tiles tiles (look-back
 * state of the cross-block scan: an 8-byte header plus 8 bytes per index
 * group of 32 tiles). */
size_t hq_encode_workspace_bytes(int64_t n_tiles);

/* Encode n_tiles bf16 tiles (Method 1-4).
 *   d_x        [n_tiles][128] bf16 bit patterns, device.
 *   d_stream   device output words, capacity cap_words; NULL = size query
 *              (only d_offsets is written).
 *   d_offsets  device [hq_num_groups(n_tiles) + 1] uint64 word offsets;
 *              always written completely (last entry = total words).
 *   d_ws       device workspace of ws_bytes >= hq_encode_workspace_bytes();
 *              zeroed by hq_encode with cudaMemsetAsync unless
 *              HQ_FLAG_WORKSPACE_READY is set.
 *   d_status   device uint32, OR-ed with HQ_ERR_{CAPACITY,TIMEOUT,RANGE}.
 * Returns HQ_OK, HQ_ERR_INVALID or HQ_ERR_CUDA.  Asynchronous. */
int hq_encode(const hq_params *p, const uint16_t *d_x, int64_t n_tiles, uint32_t *d_stream,
              uint64_t cap_words, uint64_t *d_offsets, void *d_ws, size_t ws_bytes,
              uint32_t *d_status, hq_stream_t stream);

/* Payload size of an encode without writing it (Method 3: the realized rate
 * counts Rice bits, the kept remainder bits and the unary codes of every
 * symbol; group padding and the index are not payload).  Runs the encoder in
 * size mode over the same tiles and adds their payload bits to *d_bits.
 *   d_bits     device uint64, 8-byte aligned; the caller zeroes it (calls
 *              accumulate).
 *   d_ws       as for hq_encode; d_status OR-ed with HQ_ERR_{TIMEOUT,RANGE}.
 * Returns HQ_OK, HQ_ERR_INVALID or HQ_ERR_CUDA.  Asynchronous. */
int hq_payload_bits(const hq_params *p, const uint16_t *d_x, int64_t n_tiles, uint64_t *d_bits,
                    void *d_ws, size_t ws_bytes, uint32_t *d_status, hq_stream_t stream);

/* Result of hq_calibrate. */
typedef struct hq_calibration {
  float alpha;        /* chosen alpha (fp32, as hq_params carries it) */
  int32_t rice_k;     /* chosen Rice parameter */
  double bps;         /* realized payload rate at (alpha, rice_k), bits per element */
  int32_t feasible;   /* 1 if some k in [k_min, k_max] reached the target within tol */
  int32_t evaluations;/* rate evaluations made (one size-mode encode each) */
} hq_calibration;

/* Rate calibration of alpha and the Rice parameter (Method 2: alpha is set so
 * that the codes fit the budget; Method 3: the realized rate lands within
 * about 0.01 bps of the target, k chosen per rate).  For each k in
 * [k_min, k_max]: if the rate at alpha = 2^-14 already exceeds
 * target_bps - tol/2 the k is skipped; otherwise log2(alpha) is bisected on
 * [-14, 18] (at most 60 steps, stopping once |rate - target| <= tol) and the
 * midpoint with the rate nearest the target is rounded to fp32 and evaluated
 * again; it is feasible if that rate is within tol.  The feasible k with the
 * largest alpha (least distortion) wins, ties to the smaller k.  Rates are
 * hq_payload_bits / (128 n_tiles) of the tiles given; p supplies lattice,
 * dither, seeds, signs and segments (its alpha and rice_k are ignored).
 *   d_bits     device uint64 scratch; d_status device uint32 scratch, zeroed
 *              before every evaluation (it holds the last evaluation's bits).
 * Synchronous: every evaluation is read back with cudaStreamSynchronize on
 * `stream` (the only entry point that waits on the GPU).  Returns HQ_OK (see
 * out->feasible), HQ_ERR_INVALID, or HQ_ERR_CUDA (also when a cross-block
 * wait ran out). */
int hq_calibrate(const hq_params *p, const uint16_t *d_x, int64_t n_tiles, double target_bps,
                 double tol, int k_min, int k_max, void *d_ws, size_t ws_bytes,
                 uint64_t *d_bits, uint32_t *d_status, hq_stream_t stream,
                 hq_calibration *out);

/* Decode n_tiles tiles from a stream written by hq_encode with the same
 * params (Method 1-4 inverted: unpack, Rice decode, restore stripped bits,
 * subtract dither, inverse RHT).
 *   d_stream   device words [stream_words]; a group whose index entries
 *              point outside [0, stream_words] is treated as corrupt, so a
 *              damaged index never causes a read past the buffer.
 *   d_out      [n_tiles][128], bf16 (out_kind HQ_OUT_BF16, round to nearest
 *              even) or fp32 (HQ_OUT_F32).
 * A group failing a format check decodes to zeros and sets HQ_ERR_CORRUPT.
 * Returns HQ_OK, HQ_ERR_INVALID or HQ_ERR_CUDA.  Asynchronous. */
int hq_decode(const hq_params *p, const uint32_t *d_stream, uint64_t stream_words,
              const uint64_t *d_offsets, int64_t n_tiles, void *d_out, int out_kind,
              uint32_t *d_status, hq_stream_t stream);

/* Bytes of device workspace hq_decode_qk needs (rotated queries, fp32). */
size_t hq_decode_qk_workspace_bytes(int B, int Hq);

/* Attention scores from compressed K (closing section, fused decode + MMA):
 *   scores[b][hq][t] = sum_d q[b][hq][d] * Khat[h][t][d],  h = hq / (Hq / n_kv_heads),
 * with Khat the decode of K tile h * n_tokens + t; K itself is never written.
 * The products run on the tensor cores: each query row and each key is
 * scaled by a power of two (exact) to below 1 in magnitude and split into
 * two fp16 parts (|x - hi - lo| <= 2^-22 |x| + 2^-25), the partial products
 * summed in an fp32 accumulator and the scales undone, an fp32-level result.
 *   d_q        [B][Hq][128] bf16, device.
 *   d_scores   [B][Hq][n_tokens] fp32, device.
 *   d_ws       >= hq_decode_qk_workspace_bytes(B, Hq) bytes, device.
 *   d_status   OR-ed with HQ_ERR_CORRUPT for a damaged group, HQ_ERR_TIMEOUT
 *              if a tensor-core completion wait ran out (its scores are then
 *              not written).
 * Requires Hq % n_kv_heads == 0 and every head's tiles in one sign segment
 * (tiles_per_segment a multiple of n_tokens).  Returns HQ_OK, HQ_ERR_INVALID
 * or HQ_ERR_CUDA.  Asynchronous. */
int hq_decode_qk(const hq_params *p, const uint32_t *d_k_stream, uint64_t stream_words,
                 const uint64_t *d_k_offsets, int n_kv_heads, int64_t n_tokens, const uint16_t *d_q, int B, int Hq,
                 float *d_scores, void *d_ws, size_t ws_bytes, uint32_t *d_status,
                 hq_stream_t stream);

/* Bytes of device workspace hq_decode_attention needs: the rotated queries
 * (B * Hq * 128 fp32), the scores (B * Hq * n_tokens fp32), and per chunk of
 * tokens the partial sums of the value contraction and the softmax maximum
 * and sum of each query row (sized for the smallest chunk, 4 groups of 32
 * tokens; the launch may use larger ones).  0 for invalid sizes. */
size_t hq_decode_attention_workspace_bytes(int n_kv_heads, int64_t n_tokens, int B, int Hq);

/* One decode step of attention read straight from compressed K and V
 * (closing section, fused decode + MMA; Method 4 for the KV cache):
 *   s[b][hq][t] = scale * sum_d q[b][hq][d] * Khat[h][t][d],  h = hq / (Hq / n_kv_heads)
 *   p[b][hq][.] = softmax over t of s[b][hq][.]
 *   out[b][hq][d] = sum_t p[b][hq][t] * Vhat[h][t][d]
 * with Khat / Vhat the decodes of tile h * n_tokens + t of the K / V stream
 * (each with its own params pk / pv).  Neither K nor V is written out: the
 * value side is accumulated in the lattice domain and transformed once per
 * query row; the softmax is formed per chunk of tokens (maximum and sum) and
 * the chunks are combined in a fixed order, so the result is deterministic.
 * Both contractions run on the tensor cores with fp32 accumulators: the
 * scores as in hq_decode_qk, the value sums with operands split into two tf32
 * parts (|x - hi - lo| <= 2^-22 |x|).
 *   d_q        [B][Hq][128] bf16, device.
 *   d_out      [B][Hq][128] fp32, device, 16-byte aligned.
 *   d_probs    optional [B][Hq][n_tokens] fp32 output of p (NULL: p is not
 *              formed; the scores stay in the workspace).
 *   d_ws       >= hq_decode_attention_workspace_bytes() bytes, 16-byte aligned.
 *   d_status   OR-ed with HQ_ERR_CORRUPT for a damaged group of either stream,
 *              HQ_ERR_TIMEOUT if a tensor-core completion wait ran out.
 * Requires Hq % n_kv_heads == 0 and every head's tiles in one sign segment of
 * each stream (tiles_per_segment of pk and pv multiples of n_tokens).
 * Returns HQ_OK, HQ_ERR_INVALID or HQ_ERR_CUDA.  Asynchronous. */
int hq_decode_attention(const hq_params *pk, const uint32_t *d_k_stream, uint64_t k_words,
                        const uint64_t *d_k_offsets, const hq_params *pv,
                        const uint32_t *d_v_stream, uint64_t v_words,
                        const uint64_t *d_v_offsets, int n_kv_heads, int64_t n_tokens,
                        const uint16_t *d_q, int B, int Hq, float scale, float *d_out,
                        float *d_probs, void *d_ws, size_t ws_bytes, uint32_t *d_status,
                        hq_stream_t stream);

/* Bytes of device workspace hq_decode_gemm needs: the rotated activations
 * (B * cols fp32) and one partial sum per (activation row, tile)
 * (B * rows * cols / 128 fp32).  0 for invalid sizes. */
size_t hq_decode_gemm_workspace_bytes(int64_t rows, int64_t cols, int B);

/* Product with a compressed weight matrix (Method 2: weights coded with the
 * same tile codec; closing section: decode fused with the matrix product):
 *   y[b][o] = sum_i What[o][i] * x[b][i]
 * where W [rows][cols] (cols a multiple of 128) was coded row-major, tile t
 * holding W[t / (cols/128)][128 (t % (cols/128)) ...], and What is its decode.
 * What is never written: each tile is decoded to the lattice domain and dotted
 * with the activation tile rotated once (s_dec H D x).
 *   d_x        [B][cols] bf16, device.
 *   d_y        [B][rows] fp32, device.
 *   d_ws       >= hq_decode_gemm_workspace_bytes() bytes, 16-byte aligned.
 *   d_status   OR-ed with HQ_ERR_CORRUPT for a damaged group.
 * Requires the whole matrix in one sign segment (p->tiles_per_segment >=
 * rows * cols / 128).  The sum over a row's tiles has a fixed order, so the
 * result is deterministic.  Returns HQ_OK, HQ_ERR_INVALID or HQ_ERR_CUDA.
 * Asynchronous. */
int hq_decode_gemm(const hq_params *p, const uint32_t *d_w_stream, uint64_t w_words,
                   const uint64_t *d_w_offsets, int64_t rows, int64_t cols, const uint16_t *d_x,
                   int B, float *d_y, void *d_ws, size_t ws_bytes, uint32_t *d_status,
                   hq_stream_t stream);

/* Largest n_tiles accepted by hq_encode_noalloc: 2^22 tiles (2^29 elements,
 * 1 GiB of bf16 per call). */
#define HQ_NOALLOC_MAX_TILES (1LL << 22)

/* hq_encode for callers that cannot allocate device memory.  The summary has
 * no counterpart to this entry point; it exists for deployment.  Some callers
 * may not call cudaMalloc at the point where they encode: a serving engine
 * that hands all free device memory to its own cache pool at start-up (a new
 * allocation would fail or fragment that pool), a latency-critical path where
 * cudaMalloc / cudaFree may synchronise the device, or a plugin inside a host
 * framework that owns every allocation and offers the plugin no allocator.
 * Such callers cannot provide the encoder's workspace, so this variant uses a
 * fixed scratch array compiled into the library instead (about 1 MiB, held in
 * every GPU that loads the library until the process exits).
 *   Arguments, outputs and status bits are those of hq_encode without d_ws /
 *   ws_bytes; the caller still passes (and owns) the input, the output words,
 *   the offsets and the status word.  Neither this function nor anything it
 *   calls allocates: the scratch is cleared with cudaMemsetAsync on `stream`.
 *   n_tiles > HQ_NOALLOC_MAX_TILES returns HQ_ERR_INVALID, nothing launched.
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture.  The cached address belongs to the
 *   device's current primary context: after cudaDeviceReset (or anything else
 *   that destroys that context) the address is stale, so do not call this
 *   entry point again in that process.
 *   All calls on a device share the one scratch array: calls that may overlap
 *   on the GPU (different streams without ordering between them) race and
 *   corrupt each other's scan; serialise them (one stream, or events).
 * Returns HQ_OK, HQ_ERR_INVALID or HQ_ERR_CUDA.  Asynchronous. */
int hq_encode_noalloc(const hq_params *p, const uint16_t *d_x, int64_t n_tiles,
                      uint32_t *d_stream, uint64_t cap_words, uint64_t *d_offsets,
                      uint32_t *d_status, hq_stream_t stream);

/* Host: the 128-bit sign mask of (seed, segment) -- one Philox4x32-10 call
 * (Salmon et al., SC'11) with key (seed lo, seed hi) and counter
 * (segment lo, segment hi, 0, 0x5349474E).  out[4] is host memory. */
void hq_make_signs(uint64_t seed, uint64_t segment, uint32_t out[4]);

/* Host: the sign mask of one layer of a KV cache, D XOR S_layer -- the random
 * diagonal D of the transform (Method 1, drawn once per model from seed_d,
 * segment 0) composed with the per-layer +-1 rotation S_layer (Method 4,
 * drawn from seed_s with the layer as segment).  Both are diagonal and act
 * before H, so they compose into one mask: out[i] = hq_make_signs(seed_d,
 * 0)[i] ^ hq_make_signs(seed_s, layer)[i].  out[4] is host memory. */
void hq_make_layer_signs(uint64_t seed_d, uint64_t seed_s, uint64_t layer, uint32_t out[4]);

/* Host: a static, human-readable name for a status value or bit set. */
const char *hq_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif  /* HQ_H_ */

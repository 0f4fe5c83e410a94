// hq_noalloc.cu -- hq_encode_noalloc: the encoder for callers that cannot
// allocate device memory.
//
// The encoder's only scratch is the look-back state of its cross-block scan
// (a ticket counter plus 8 bytes per index group of 32 tiles).  hq_encode takes
// that scratch from the caller; this entry point instead uses a fixed array
// compiled into the library, so neither the library nor the caller allocates
// anything.  The array lives in every GPU's memory from the moment the
// library's module is loaded on that GPU until the process exits.
#include <mutex>

#include <cuda_runtime.h>

#include "hq_device.cuh"
#include "hq_internal.h"

namespace {

// 8-byte ticket header + 8 bytes of look-back state per encoder block (one
// block per kGroupTiles tiles, the constant the encoder itself uses) for
// HQ_NOALLOC_MAX_TILES tiles, rounded up to 256 bytes.
constexpr size_t kNoallocScratchBytes =
    ((8 + 8 * (size_t)((HQ_NOALLOC_MAX_TILES + hq::kGroupTiles - 1) / hq::kGroupTiles)) + 255) /
    256 * 256;

static __device__ __align__(256) unsigned char g_encode_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mutex;
void *g_scratch_address[kMaxDevices] = {};

// Device address of g_encode_scratch on the current device.  The symbol's
// name is only a host-side stand-in, so its address is looked up once per
// device (with that device current) and cached.
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_address[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_encode_scratch) != cudaSuccess || ptr == nullptr)
      return HQ_ERR_CUDA;
    g_scratch_address[dev] = ptr;
  }
  *out = g_scratch_address[dev];
  return HQ_OK;
}

}  // namespace

extern "C" int hq_encode_noalloc(const hq_params *p, const uint16_t *d_x, int64_t n_tiles,
                                 uint32_t *d_stream, uint64_t cap_words, uint64_t *d_offsets,
                                 uint32_t *d_status, hq_stream_t stream) {
  if (!p || n_tiles < 0 || n_tiles > HQ_NOALLOC_MAX_TILES) return HQ_ERR_INVALID;
  void *scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != HQ_OK) return rc;
  size_t need = hq_encode_workspace_bytes(n_tiles);
  if (need > kNoallocScratchBytes) return HQ_ERR_INVALID;
  // The scratch keeps whatever the previous call left in it: always let
  // hq_encode clear it (ticket counter and look-back flags must start at 0).
  hq_params q = *p;
  q.flags &= ~HQ_FLAG_WORKSPACE_READY;
  return hq_encode(&q, d_x, n_tiles, d_stream, cap_words, d_offsets, scratch,
                   kNoallocScratchBytes, d_status, stream);
}

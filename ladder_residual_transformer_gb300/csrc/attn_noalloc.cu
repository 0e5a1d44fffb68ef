// Decode attention for callers that cannot allocate device memory.
//
// ladder_attention_decode needs a scratch buffer for its per-split partial
// results, which the caller normally allocates.  Some callers have no way to do
// that: code that runs while another component is capturing a CUDA graph
// (allocation calls are not allowed inside a capture), plugins embedded in a
// host framework that owns every device allocation, or latency-critical loops
// where an allocation may stall on a device-wide synchronisation.  This entry
// point keeps the scratch in a file-scope device array instead, so it allocates
// nothing.  The array is part of the loaded module: every GPU on which the
// library runs this code holds it until the process exits.
#include "ladder.h"
#include "internal.cuh"

#include <cstdio>
#include <mutex>
#include <string>

namespace ladder {
int set_error(int code, const char* msg);
}

using namespace ladder;

namespace {

constexpr size_t kStaticScratchBytes = LADDER_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Partials of the split attention: [B][n_q][nsplit][head_dim] fp32, then
// [B][n_q][nsplit][2] fp32 (running max, running sum) at a 256-byte boundary.
static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(LADDER_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return set_error(LADDER_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess || !p) return set_error(LADDER_ERR_CUDA, "cudaGetSymbolAddress(g_attn_scratch) failed");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LADDER_OK;
}

}  // namespace

extern "C" int ladder_attention_decode_noalloc(const float* q, const void* kv_layer, int32_t kv_dtype,
                                               const int32_t* block_table, int32_t max_pages_per_seq,
                                               const int32_t* positions, int32_t B, int32_t n_q_heads,
                                               int32_t n_kv_heads, int32_t head_dim, int32_t page_size, float scale,
                                               int32_t max_position, float* out, ladder_stream_t stream) {
  if (B <= 0 || n_q_heads <= 0 || head_dim <= 0 || max_position < 0)
    return set_error(LADDER_ERR_INVALID, "B, n_q_heads, head_dim must be positive and max_position >= 0");
  // the same sizing rule as the scratch-taking entry point, from the one place that defines it
  const size_t need = ladder_attention_decode_scratch_bytes(B, n_q_heads, head_dim, max_position);
  if (need > kStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "attention needs %zu bytes of scratch, more than the %zu-byte static array of the no-allocation entry "
             "point: use ladder_attention_decode with a caller buffer",
             need, kStaticScratchBytes);
    return set_error(LADDER_ERR_CAPACITY, msg);
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  // Every partial that the combine step reads is written earlier in the same
  // call, so nothing in the array has to start at zero.
  return ladder_attention_decode(q, kv_layer, kv_dtype, block_table, max_pages_per_seq, positions, B, n_q_heads,
                                 n_kv_heads, head_dim, page_size, scale, max_position, out, scratch,
                                 kStaticScratchBytes, stream);
}

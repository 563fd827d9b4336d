// Allocation-free decode attention: oscar_decode_attention with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory (an engine whose memory is fully reserved up front, or
// a decode loop that must not block on the allocator), the workspace of oscar_decode_attention (rotated
// queries and split-K partials) comes from the file-scope array below instead of from the caller.
#include <cstdio>
#include <mutex>

#include "oscar_internal.cuh"
#include "kernels.h"

namespace {

// The scratch itself.  In host code this name only stands in for the symbol; its device address is
// looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[OSCAR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

}  // namespace

extern "C" oscar_status_t oscar_decode_attention_noalloc(const oscar_pool *pool, const oscar_bf16 *q, float *out,
                                                         float softmax_scale, oscar_stream_t stream) {
  char msg[256];
  size_t need = 0;
  oscar_status_t st = oscar_decode_workspace_size(pool, 0, &need);  // validates the pool
  if (st != OSCAR_OK) return st;
  if (need > OSCAR_NOALLOC_SCRATCH_BYTES) {
    snprintf(msg, sizeof msg,
             "decode_attention_noalloc: this pool needs %zu bytes of scratch, more than the %u-byte static "
             "array; use oscar_decode_attention with a caller workspace",
             need, (unsigned)OSCAR_NOALLOC_SCRATCH_BYTES);
    oscar::set_last_error(msg);
    return OSCAR_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "decode_attention_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    oscar::set_last_error(msg);
    return OSCAR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof msg, "decode_attention_noalloc: device %d beyond the %d supported", dev, kMaxDevices);
    oscar::set_last_error(msg);
    return OSCAR_ERR_UNSUPPORTED;
  }
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {  // set-up, once per device, with that device current
      e = cudaGetSymbolAddress(&g_scratch_addr[dev], g_noalloc_scratch);
      if (e != cudaSuccess) {
        g_scratch_addr[dev] = nullptr;
        snprintf(msg, sizeof msg, "decode_attention_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        oscar::set_last_error(msg);
        return OSCAR_ERR_CUDA;
      }
    }
    scratch = g_scratch_addr[dev];
  }
  return oscar_decode_attention(pool, q, out, softmax_scale, 0, scratch, OSCAR_NOALLOC_SCRATCH_BYTES, stream);
}

// Allocation-free decode attention: oscar_decode_attention with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory (an engine whose memory is fully reserved up front, or
// a decode loop that must not block on the allocator), the workspace of oscar_decode_attention (rotated
// queries and split-K partials) comes from the file-scope array below instead of from the caller.
#include <cstdio>
#include <mutex>
#include <utility>

#include <cuda.h>

#include "oscar_internal.cuh"
#include "kernels.h"

namespace {

// The scratch itself.  In host code this name only stands in for the symbol; its device address is
// looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[OSCAR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// The looked-up address per device, with the identifier of the context it belongs to: a device reset
// (cudaDeviceReset) ends the context and the array gets a new address in the next one, so the address
// is looked up again whenever the current context is not the one it was found in.
struct ScratchAddr {
  unsigned long long ctx_id = 0;
  void *addr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

// Identifier of the calling thread's current CUDA context (driver entry points cuCtxGetCurrent and
// cuCtxGetId, looked up once); 0 if the driver does not provide them.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static const std::pair<GetCurrent, GetId> fns = [] {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess)
      a = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      b = nullptr;
    return std::make_pair(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (fns.first == nullptr || fns.second == nullptr || fns.first(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      fns.second(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

}  // namespace

extern "C" oscar_status_t oscar_decode_attention_noalloc(const oscar_pool *pool, const oscar_bf16 *q, float *out,
                                                         float softmax_scale, oscar_stream_t stream) {
  char msg[256];
  size_t need = 0;
  oscar_status_t st = oscar::decode_workspace_min(pool, &need);  // validates the pool
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
    // (the size query above has already made the runtime create the device's context)
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddr &slot = g_scratch_addr[dev];
    if (slot.addr == nullptr || slot.ctx_id != ctx) {  // set-up, once per device (and context), device current
      void *addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess) {
        slot = ScratchAddr{};
        snprintf(msg, sizeof msg, "decode_attention_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        oscar::set_last_error(msg);
        return OSCAR_ERR_CUDA;
      }
      slot.addr = addr;
      slot.ctx_id = ctx;
    }
    scratch = slot.addr;
  }
  return oscar_decode_attention(pool, q, out, softmax_scale, 0, scratch, OSCAR_NOALLOC_SCRATCH_BYTES, stream);
}

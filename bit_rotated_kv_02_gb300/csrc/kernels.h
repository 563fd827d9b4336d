// Launchers shared between the API layer and the kernel translation units (internal).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "oscar_internal.cuh"

namespace oscar {

// Per-thread profiling events armed by oscar_profile_events (api.cu); launchers record them around the
// kernel of the matching kind and disarm.
struct ProfileSlot {
  cudaEvent_t start = nullptr, stop = nullptr;
};
ProfileSlot &profile_slot(int which);
inline void profile_begin(int which, cudaStream_t s) {
  ProfileSlot &p = profile_slot(which);
  if (p.start) cudaEventRecord(p.start, s);
}
inline void profile_end(int which, cudaStream_t s) {
  ProfileSlot &p = profile_slot(which);
  if (p.stop) cudaEventRecord(p.stop, s);
  p.start = p.stop = nullptr;
}

// A value computed once per device (SM count x resident CTAs of a kernel) and kept for the process:
// `slots` holds one entry per device index (0 = not yet computed); `compute` runs with that device
// current.  Concurrent first calls from several host threads compute the same value; the store is atomic.
constexpr int kMaxDevices = 64;
template <class F>
int per_device(std::atomic<int> (&slots)[kMaxDevices], F compute) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return compute(dev);
  int v = slots[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    v = compute(dev);
    slots[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Sets the calling thread's oscar_last_error_string() (api.cu).
void set_last_error(const char *msg);

// Launch with programmatic stream serialization (the kernel must start with pdl_wait()): its blocks
// may be scheduled while the previous kernel of the stream finishes, hiding the launch gap.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// quantize.cu
cudaError_t launch_demote(const PoolArgs &p, const int32_t *mask, int mode, const uint16_t *k_new,
                          const uint16_t *v_new, cudaStream_t s);
cudaError_t launch_quantize_rows(int64_t n, int Hkv, int g, const uint16_t *x, int64_t x_row_stride, const float *R32,
                                 const float *clip, uint8_t *codes, uint16_t *scale, uint16_t *zero,
                                 const int32_t *pt, int num_pages, uint32_t *err, uint32_t *stats, cudaStream_t s);
// The same with codebook levels cb [Hkv][4] (CUDA-core rotation; the tensor-core kernel serves the uniform levels).
cudaError_t launch_quantize_rows_cb(int64_t n, int Hkv, int g, const uint16_t *x, int64_t x_row_stride,
                                    const float *R32, const float *clip, const float *cb, uint8_t *codes,
                                    uint16_t *scale, uint16_t *zero, const int32_t *pt, int num_pages, uint32_t *err,
                                    uint32_t *stats, cudaStream_t s);
cudaError_t launch_prefill(const PoolArgs &p, int b, int64_t L, const uint16_t *k, const uint16_t *v, uint32_t *stats,
                           cudaStream_t s, int skip = 0);
// codebook.cu: Lloyd-Max levels [Hkv][4] from calibration rows x [n][Hkv][D] (workspace: lloyd_ws_bytes).
size_t lloyd_ws_bytes(int64_t n, int Hkv);
cudaError_t launch_lloyd_max(int64_t n, int Hkv, int g, const uint16_t *x, const float *R32, const float *clip,
                             int iters, float *cb_out, void *ws, cudaStream_t s);

// decode.cu
constexpr int PART_STRIDE = D + 4;  // one partial: o[128], m, l, pad
size_t decode_ws_bytes(const PoolArgs &p, int splits);
cudaError_t launch_decode(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, int splits, float *ws,
                          cudaStream_t s);

// decode_v1.cu (tensor-core path, group size 128)
// Workspace bytes: dyn = false the minimum, dyn = true with the dynamic tail of the history split (its
// partial slots and chunk counter); a launch with dyn uses that tail.
size_t v1_ws_bytes(const PoolArgs &p, bool dyn);
cudaError_t launch_decode_v1(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                             cudaStream_t s, bool dyn);
// The decode step for group size 128: the query rotation, the attention kernel and the merge, which
// performs the demotion and the append.
cudaError_t launch_step_v1(const PoolArgs &p, const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q,
                           float *out, float sm_scale, float *ws, cudaStream_t s, bool dyn);

// The merge kernel of decode_v1.cu (LSE merge, o . R_v^T, normalisation; k_new != NULL: the decode-step form
// with the append and the counter update) over partial slots in its layout.
// The smallest decode workspace a call on this pool accepts (api.cu; validates the pool).
oscar_status_t decode_workspace_min(const oscar_pool *pool, size_t *bytes);

// dyn: the history partials include the dynamic tail's (decode_v1.cu's attention with dyn).
cudaError_t launch_merge_v1(const PoolArgs &p, const float *part, int n_hist, float *out, const uint16_t *k_new,
                            const uint16_t *v_new, cudaStream_t s, bool dyn = false);

// decode_tc.cu (tcgen05 path, uniform levels, group sizes 32, 64, 128): history CTAs (one per SM), workspace
// bytes, and the launch (query rotation + operand images, history, BF16 + demotion, merge); k_new != NULL:
// the decode-step form.
int tc_hist_ctas(const PoolArgs &p);
size_t tc_ws_bytes(const PoolArgs &p);
cudaError_t launch_decode_tc(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                             cudaStream_t s, const uint16_t *k_new = nullptr, const uint16_t *v_new = nullptr);

// quant_tc.cu: cuTensorMapEncodeTiled from the driver (nullptr if the driver lacks it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// decode_bf16.cu (the BF16 paged cache that INT2 decoding is compared against)
struct CacheArgs {
  int B, Hq, Hkv, num_pages, max_pages;
  uint16_t *k_pages, *v_pages;  // bf16 [num_pages][Hkv][64][D]
  int32_t *page_table, *seq_len;
  uint32_t *err;
};
int bf16_attn_ctas(const CacheArgs &c);
size_t bf16_ws_bytes(const CacheArgs &c);
// k_new != nullptr: append the new token first (one more launch, chained).
cudaError_t launch_bf16_decode(const CacheArgs &c, const uint16_t *q, float *out, float sm_scale, float *ws,
                               cudaStream_t s, const uint16_t *k_new = nullptr, const uint16_t *v_new = nullptr);
cudaError_t launch_bf16_append(const CacheArgs &c, const uint16_t *k_new, const uint16_t *v_new, cudaStream_t s);
cudaError_t launch_bf16_prefill(const CacheArgs &c, int seq, int len, const uint16_t *k, const uint16_t *v,
                                cudaStream_t s);

// rotation.cu
size_t rotation_ws_bytes(int d);
cudaError_t launch_make_rotation(int d, int mode, const double *M, double *R64, float *R32, void *ws,
                                 cudaStream_t s);
cudaError_t launch_cov_k(int64_t T, int heads, int d, const uint16_t *Q, double *C, cudaStream_t s);
size_t cov_v_ws_bytes(int64_t T, int d);
cudaError_t launch_cov_v(int64_t T, int heads, int d, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                         double scale, double *C, void *ws, cudaStream_t s);

}  // namespace oscar

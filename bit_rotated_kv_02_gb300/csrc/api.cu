// C ABI of liboscar: host-side validation, workspace sizing and kernel launches.
// Every entry point validates its arguments before any launch and reports failures through its
// return status and oscar_last_error_string().
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "oscar_internal.cuh"
#include "kernels.h"

using namespace oscar;

namespace {

thread_local std::string g_last_error;
thread_local ProfileSlot g_profile[2];

oscar_status_t fail(oscar_status_t st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

oscar_status_t cuda_status(cudaError_t e, const char *where) {
  if (e == cudaSuccess) return OSCAR_OK;
  return fail(OSCAR_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool supported_group(int g) { return g == 32 || g == 64 || g == 128; }

oscar_status_t check_pool(const oscar_pool *pool, PoolArgs &a) {
  if (pool == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "pool is NULL");
  const oscar_pool &p = *pool;
  if (p.head_dim != OSCAR_HEAD_DIM) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d (only 128)", p.head_dim);
  if (!supported_group(p.group_size)) return fail(OSCAR_ERR_UNSUPPORTED, "group_size %d (32, 64 or 128)", p.group_size);
  if (p.batch <= 0 || p.num_kv_heads <= 0 || p.num_q_heads <= 0)
    return fail(OSCAR_ERR_INVALID_ARG, "batch/heads must be positive");
  if (p.num_q_heads % p.num_kv_heads != 0)
    return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", p.num_q_heads, p.num_kv_heads);
  const int G = p.num_q_heads / p.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(OSCAR_ERR_UNSUPPORTED, "GQA ratio %d (1, 2, 4 or 8)", G);
  if (p.num_pages < 0 || p.max_pages < 0) return fail(OSCAR_ERR_INVALID_ARG, "negative page counts");
  if ((int64_t)p.max_pages * OSCAR_PAGE_TOKENS > (int64_t)1 << 30)
    return fail(OSCAR_ERR_INVALID_ARG, "max_pages %d too large", p.max_pages);
  const void *ptrs[] = {p.sink_k, p.sink_v, p.recent_k, p.recent_v, p.codes_k, p.codes_v, p.scale_k, p.zero_k,
                        p.scale_v, p.zero_v, p.page_table, p.sink_len, p.hist_len, p.recent_start, p.recent_len,
                        p.R_k, p.R_v, p.clip_k, p.clip_v, p.err, p.sync};
  const char *names[] = {"sink_k", "sink_v", "recent_k", "recent_v", "codes_k", "codes_v", "scale_k", "zero_k",
                         "scale_v", "zero_v", "page_table", "sink_len", "hist_len", "recent_start", "recent_len",
                         "R_k", "R_v", "clip_k", "clip_v", "err", "sync"};
  for (size_t i = 0; i < sizeof(ptrs) / sizeof(ptrs[0]); ++i) {
    const bool pool_storage = i >= 4 && i <= 10;  // history arrays may be NULL only without pages
    if (ptrs[i] == nullptr && !(pool_storage && (p.num_pages == 0 || p.max_pages == 0)))
      return fail(OSCAR_ERR_INVALID_ARG, "pool.%s is NULL", names[i]);
  }
  if ((reinterpret_cast<uintptr_t>(p.codes_k) | reinterpret_cast<uintptr_t>(p.codes_v) |
       reinterpret_cast<uintptr_t>(p.sink_k) | reinterpret_cast<uintptr_t>(p.sink_v) |
       reinterpret_cast<uintptr_t>(p.recent_k) | reinterpret_cast<uintptr_t>(p.recent_v) |
       reinterpret_cast<uintptr_t>(p.R_k) | reinterpret_cast<uintptr_t>(p.R_v)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "pool arrays must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(p.scale_k) | reinterpret_cast<uintptr_t>(p.zero_k) |
       reinterpret_cast<uintptr_t>(p.scale_v) | reinterpret_cast<uintptr_t>(p.zero_v)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "pool scale/zero arrays must be 16-byte aligned");
  a.B = p.batch; a.Hq = p.num_q_heads; a.Hkv = p.num_kv_heads; a.d = p.head_dim; a.g = p.group_size;
  a.ng = p.head_dim / p.group_size; a.num_pages = p.num_pages; a.max_pages = p.max_pages;
  a.sink_k = p.sink_k; a.sink_v = p.sink_v; a.recent_k = p.recent_k; a.recent_v = p.recent_v;
  a.codes_k = p.codes_k; a.codes_v = p.codes_v; a.scale_k = p.scale_k; a.zero_k = p.zero_k;
  a.scale_v = p.scale_v; a.zero_v = p.zero_v; a.page_table = p.page_table; a.sink_len = p.sink_len;
  a.hist_len = p.hist_len; a.recent_start = p.recent_start; a.recent_len = p.recent_len;
  if ((reinterpret_cast<uintptr_t>(p.codebook_k) | reinterpret_cast<uintptr_t>(p.codebook_v)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "pool codebooks must be 16-byte aligned");
  a.R_k = p.R_k; a.R_v = p.R_v; a.clip_k = p.clip_k; a.clip_v = p.clip_v; a.err = p.err; a.sync = p.sync;
  a.cb_k = p.codebook_k; a.cb_v = p.codebook_v;
  return OSCAR_OK;
}

oscar_status_t check_cache(const oscar_bf16_cache *cache, CacheArgs &a) {
  if (cache == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  const oscar_bf16_cache &c = *cache;
  if (c.head_dim != OSCAR_HEAD_DIM) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d (only 128)", c.head_dim);
  if (c.batch <= 0 || c.num_kv_heads <= 0 || c.num_q_heads <= 0)
    return fail(OSCAR_ERR_INVALID_ARG, "batch/heads must be positive");
  if (c.num_q_heads % c.num_kv_heads != 0)
    return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", c.num_q_heads, c.num_kv_heads);
  const int G = c.num_q_heads / c.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(OSCAR_ERR_UNSUPPORTED, "GQA ratio %d (1, 2, 4 or 8)", G);
  if (c.num_pages <= 0 || c.max_pages <= 0) return fail(OSCAR_ERR_INVALID_ARG, "page counts must be positive");
  if ((int64_t)c.max_pages * OSCAR_PAGE_TOKENS > (int64_t)1 << 30)
    return fail(OSCAR_ERR_INVALID_ARG, "max_pages %d too large", c.max_pages);
  if ((int64_t)c.num_pages * c.num_kv_heads * OSCAR_PAGE_TOKENS >= (int64_t)1 << 31)
    return fail(OSCAR_ERR_INVALID_ARG, "num_pages * Hkv * 64 must stay below 2^31");
  if (c.k_pages == nullptr || c.v_pages == nullptr || c.page_table == nullptr || c.seq_len == nullptr ||
      c.err == nullptr)
    return fail(OSCAR_ERR_INVALID_ARG, "cache pointer is NULL");
  if ((reinterpret_cast<uintptr_t>(c.k_pages) | reinterpret_cast<uintptr_t>(c.v_pages)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "cache page arrays must be 16-byte aligned");
  a.B = c.batch; a.Hq = c.num_q_heads; a.Hkv = c.num_kv_heads; a.num_pages = c.num_pages; a.max_pages = c.max_pages;
  a.k_pages = c.k_pages; a.v_pages = c.v_pages; a.page_table = c.page_table; a.seq_len = c.seq_len; a.err = c.err;
  return OSCAR_OK;
}

int auto_splits(const PoolArgs &a) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // the CUDA-core history kernel is latency bound: about 16 CTAs of 128 threads per SM's worth of splits
  // (measured on mixed long-context batches: 2 per SM 4.6 ms, 16 per SM 2.1 ms, 64 per SM 2.5 ms)
  const int units = a.B * a.Hkv;
  int s = (16 * sms + units - 1) / units;
  if (s > a.max_pages) s = a.max_pages;
  return s < 1 ? 1 : s;
}

}  // namespace

namespace oscar {
ProfileSlot &profile_slot(int which) { return g_profile[which & 1]; }
void set_last_error(const char *msg) { g_last_error = msg; }
}  // namespace oscar

extern "C" {

oscar_status_t oscar_profile_events(int32_t which, void *start, void *stop) {
  if (which != OSCAR_PROFILE_HISTORY && which != OSCAR_PROFILE_DEMOTE)
    return fail(OSCAR_ERR_INVALID_ARG, "profile kind %d", which);
  if ((start == nullptr) != (stop == nullptr)) return fail(OSCAR_ERR_INVALID_ARG, "give both events or neither");
  g_profile[which].start = static_cast<cudaEvent_t>(start);
  g_profile[which].stop = static_cast<cudaEvent_t>(stop);
  return OSCAR_OK;
}

const char *oscar_last_error_string(void) { return g_last_error.c_str(); }

const char *oscar_version(void) { return "oscar-gb300 0.1 (sm_103a)"; }

size_t oscar_make_rotation_workspace_size(int32_t d) { return (d > 0) ? rotation_ws_bytes(d) : 0; }

oscar_status_t oscar_make_rotation(int32_t d, int32_t mode, const double *M, double *R64, float *R32, void *ws,
                                   size_t ws_bytes, oscar_stream_t stream) {
  if (d < 2 || d > OSCAR_HEAD_DIM || (d & (d - 1)) != 0)
    return fail(OSCAR_ERR_UNSUPPORTED, "d %d must be a power of two in [2, 128]", d);
  if (mode != OSCAR_ROT_HAAR && mode != OSCAR_ROT_COVARIANCE) return fail(OSCAR_ERR_INVALID_ARG, "mode %d", mode);
  if (M == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "M is NULL");
  if (R64 == nullptr && R32 == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "R64 and R32 are both NULL");
  if (ws == nullptr || ws_bytes < rotation_ws_bytes(d))
    return fail(OSCAR_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, rotation_ws_bytes(d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  oscar_status_t st = cuda_status(launch_make_rotation(d, mode, M, R64, R32, ws, s), "make_rotation launch");
  if (st != OSCAR_OK) return st;
  if ((st = cuda_status(cudaStreamSynchronize(s), "make_rotation")) != OSCAR_OK) return st;
  if (mode == OSCAR_ROT_COVARIANCE) {
    double status[2];
    const double *sp = static_cast<const double *>(ws) + (size_t)d * d;
    if ((st = cuda_status(cudaMemcpy(status, sp, sizeof status, cudaMemcpyDeviceToHost), "make_rotation status")) !=
        OSCAR_OK)
      return st;
    if (status[0] != 1.0) return fail(OSCAR_ERR_NUMERIC, "Jacobi eigensolver did not converge (%g sweeps)", status[1]);
  }
  return OSCAR_OK;
}

oscar_status_t oscar_calib_covariance_k(int64_t T, int32_t heads, int32_t d, const oscar_bf16 *Q, double *C,
                                        oscar_stream_t stream) {
  if (T <= 0 || heads <= 0 || d <= 0 || d > OSCAR_HEAD_DIM) return fail(OSCAR_ERR_INVALID_ARG, "bad sizes");
  if (Q == nullptr || C == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "NULL pointer");
  return cuda_status(launch_cov_k(T, heads, d, Q, C, static_cast<cudaStream_t>(stream)), "calib_covariance_k");
}

size_t oscar_calib_covariance_v_workspace_size(int64_t T, int32_t heads, int32_t d) {
  (void)heads;
  return (T > 0 && d > 0) ? cov_v_ws_bytes(T, d) : 0;
}

oscar_status_t oscar_calib_covariance_v(int64_t T, int32_t heads, int32_t d, const oscar_bf16 *Q, const oscar_bf16 *K,
                                        const oscar_bf16 *V, double softmax_scale, double *C, void *ws,
                                        size_t ws_bytes, oscar_stream_t stream) {
  if (T <= 0 || T > (1 << 16) || heads <= 0 || d <= 0 || d > OSCAR_HEAD_DIM)
    return fail(OSCAR_ERR_INVALID_ARG, "bad sizes");
  if (Q == nullptr || K == nullptr || V == nullptr || C == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "NULL pointer");
  if (!(softmax_scale > 0.0)) return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be > 0");
  if (ws == nullptr || ws_bytes < cov_v_ws_bytes(T, d))
    return fail(OSCAR_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, cov_v_ws_bytes(T, d));
  return cuda_status(launch_cov_v(T, heads, d, Q, K, V, softmax_scale, C, ws, static_cast<cudaStream_t>(stream)),
                     "calib_covariance_v");
}

oscar_status_t oscar_quantize_kv(int64_t n_tokens, int32_t num_kv_heads, int32_t head_dim, int32_t group_size,
                                 const oscar_bf16 *x, const float *R32, const float *clip, uint8_t *codes,
                                 oscar_bf16 *scale, oscar_bf16 *zero, uint32_t *stats, oscar_stream_t stream) {
  if (head_dim != OSCAR_HEAD_DIM) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d (only 128)", head_dim);
  if (!supported_group(group_size)) return fail(OSCAR_ERR_UNSUPPORTED, "group_size %d", group_size);
  if (n_tokens < 0 || num_kv_heads <= 0) return fail(OSCAR_ERR_INVALID_ARG, "bad sizes");
  if (n_tokens == 0) return OSCAR_OK;
  if (x == nullptr || R32 == nullptr || clip == nullptr || codes == nullptr || scale == nullptr || zero == nullptr)
    return fail(OSCAR_ERR_INVALID_ARG, "NULL pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(R32) | reinterpret_cast<uintptr_t>(codes)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "x, R32 and codes must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(scale) | reinterpret_cast<uintptr_t>(zero)) & 7u)
    return fail(OSCAR_ERR_INVALID_ARG, "scale and zero must be 8-byte aligned");
  return cuda_status(launch_quantize_rows(n_tokens, num_kv_heads, group_size, x, (int64_t)num_kv_heads * head_dim, R32,
                                          clip, codes, scale, zero, nullptr, 0, nullptr, stats,
                                          static_cast<cudaStream_t>(stream)),
                     "quantize_kv");
}

oscar_status_t oscar_quantize_kv_codebook(int64_t n_tokens, int32_t num_kv_heads, int32_t head_dim,
                                          int32_t group_size, const oscar_bf16 *x, const float *R32,
                                          const float *clip, const float *codebook, uint8_t *codes,
                                          oscar_bf16 *scale, oscar_bf16 *zero, uint32_t *stats,
                                          oscar_stream_t stream) {
  if (head_dim != OSCAR_HEAD_DIM) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d (only 128)", head_dim);
  if (!supported_group(group_size)) return fail(OSCAR_ERR_UNSUPPORTED, "group_size %d", group_size);
  if (n_tokens < 0 || num_kv_heads <= 0) return fail(OSCAR_ERR_INVALID_ARG, "bad sizes");
  if (n_tokens == 0) return OSCAR_OK;
  if (x == nullptr || R32 == nullptr || clip == nullptr || codebook == nullptr || codes == nullptr ||
      scale == nullptr || zero == nullptr)
    return fail(OSCAR_ERR_INVALID_ARG, "NULL pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(R32) | reinterpret_cast<uintptr_t>(codes) |
       reinterpret_cast<uintptr_t>(codebook)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "x, R32, codebook and codes must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(scale) | reinterpret_cast<uintptr_t>(zero)) & 7u)
    return fail(OSCAR_ERR_INVALID_ARG, "scale and zero must be 8-byte aligned");
  return cuda_status(launch_quantize_rows_cb(n_tokens, num_kv_heads, group_size, x, (int64_t)num_kv_heads * head_dim,
                                             R32, clip, codebook, codes, scale, zero, nullptr, 0, nullptr, stats,
                                             static_cast<cudaStream_t>(stream)),
                     "quantize_kv_codebook");
}

oscar_status_t oscar_lloyd_max_workspace_size(int64_t n, int32_t num_kv_heads, size_t *bytes) {
  if (bytes == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "bytes is NULL");
  if (n < 0 || num_kv_heads <= 0) return fail(OSCAR_ERR_INVALID_ARG, "bad sizes");
  *bytes = lloyd_ws_bytes(n, num_kv_heads);
  return OSCAR_OK;
}

oscar_status_t oscar_lloyd_max_codebook(int64_t n, int32_t num_kv_heads, int32_t head_dim, int32_t group_size,
                                        const oscar_bf16 *x, const float *R32, const float *clip,
                                        int32_t max_iters, float *codebook, void *ws, size_t ws_bytes,
                                        oscar_stream_t stream) {
  if (head_dim != OSCAR_HEAD_DIM) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d (only 128)", head_dim);
  if (!supported_group(group_size)) return fail(OSCAR_ERR_UNSUPPORTED, "group_size %d", group_size);
  if (n < 0 || num_kv_heads <= 0 || max_iters < 0) return fail(OSCAR_ERR_INVALID_ARG, "bad sizes");
  if (codebook == nullptr || (n > 0 && (x == nullptr || R32 == nullptr || clip == nullptr)))
    return fail(OSCAR_ERR_INVALID_ARG, "NULL pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(R32) | reinterpret_cast<uintptr_t>(ws)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "x, R32 and ws must be 16-byte aligned");
  const size_t need = lloyd_ws_bytes(n, num_kv_heads);
  if (need > 0 && (ws == nullptr || ws_bytes < need))
    return fail(OSCAR_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  return cuda_status(launch_lloyd_max(n, num_kv_heads, group_size, x, R32, clip, max_iters, codebook, ws,
                                      static_cast<cudaStream_t>(stream)),
                     "lloyd_max_codebook");
}

oscar_status_t oscar_prefill_pool(const oscar_pool *pool, int32_t seq, int64_t len, const oscar_bf16 *k,
                                  const oscar_bf16 *v, uint32_t *stats, oscar_stream_t stream) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  if (seq < 0 || seq >= a.B) return fail(OSCAR_ERR_INVALID_ARG, "seq %d outside [0, %d)", seq, a.B);
  if (len < 0) return fail(OSCAR_ERR_INVALID_ARG, "negative length");
  const int64_t hist = len > OSCAR_SINK_TOKENS + OSCAR_RECENT_TOKENS ? len - OSCAR_SINK_TOKENS - OSCAR_RECENT_TOKENS : 0;
  if (hist > (int64_t)a.max_pages * OSCAR_PAGE_TOKENS)
    return fail(OSCAR_ERR_INVALID_ARG, "history of %lld tokens exceeds max_pages*64", (long long)hist);
  if (len > 0 && (k == nullptr || v == nullptr)) return fail(OSCAR_ERR_INVALID_ARG, "k/v NULL");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  return cuda_status(launch_prefill(a, seq, len, k, v, stats, static_cast<cudaStream_t>(stream)), "prefill_pool");
}

oscar_status_t oscar_prefill_pool_shared(const oscar_pool *pool, int32_t seq, int64_t len, const oscar_bf16 *k,
                                         const oscar_bf16 *v, int32_t shared_pages, uint32_t *stats,
                                         oscar_stream_t stream) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  if (seq < 0 || seq >= a.B) return fail(OSCAR_ERR_INVALID_ARG, "seq %d outside [0, %d)", seq, a.B);
  if (len < 0) return fail(OSCAR_ERR_INVALID_ARG, "negative length");
  const int64_t hist = len > OSCAR_SINK_TOKENS + OSCAR_RECENT_TOKENS ? len - OSCAR_SINK_TOKENS - OSCAR_RECENT_TOKENS : 0;
  if (hist > (int64_t)a.max_pages * OSCAR_PAGE_TOKENS)
    return fail(OSCAR_ERR_INVALID_ARG, "history of %lld tokens exceeds max_pages*64", (long long)hist);
  if (shared_pages < 0 || (int64_t)shared_pages * OSCAR_PAGE_TOKENS > hist)
    return fail(OSCAR_ERR_INVALID_ARG, "shared_pages %d outside [0, %lld] (whole history pages only)", shared_pages,
                (long long)(hist / OSCAR_PAGE_TOKENS));
  if (len > 0 && (k == nullptr || v == nullptr)) return fail(OSCAR_ERR_INVALID_ARG, "k/v NULL");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  return cuda_status(launch_prefill(a, seq, len, k, v, stats, static_cast<cudaStream_t>(stream), shared_pages),
                     "prefill_pool_shared");
}

oscar_status_t oscar_demote(const oscar_pool *pool, const int32_t *mask, oscar_stream_t stream) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  return cuda_status(launch_demote(a, mask, mask ? 1 : 0, nullptr, nullptr, static_cast<cudaStream_t>(stream)),
                     "demote");
}

// The per-call inputs and outputs (q, k_new, v_new, out) are read and written by the kernels themselves: each
// must be device (or managed) memory, or page-locked host memory mapped into the device's address space at
// the same address, which the kernels then read and write over the host link.  Anything else (pageable
// host memory, a bad pointer) is refused here, before any launch.
static bool device_accessible(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged: return true;
    case cudaMemoryTypeHost: return at.devicePointer == p;
    default: return false;
  }
}
// The last pointers this thread found reachable (decode loops pass the same buffers every step; the
// attribute query costs host time comparable to a short step).  A freed and re-allocated pinned buffer keeps
// its verdict only if the new allocation at that address is pinned too or the system lets the device reach
// pageable memory (GB300 with its coherent host link does).
static bool device_accessible_cached(const void *p) {
  constexpr int N = 8;
  static thread_local const void *seen[N] = {};
  static thread_local int next = 0;
  for (int i = 0; i < N; ++i)
    if (seen[i] == p) return true;
  if (!device_accessible(p)) return false;
  seen[next] = p;
  next = (next + 1) % N;
  return true;
}
static oscar_status_t check_io(const void *p, const char *name) {
  if (!device_accessible_cached(p))
    return fail(OSCAR_ERR_INVALID_ARG, "%s is neither device memory nor page-locked host memory mapped at the same "
                "address", name);
  return OSCAR_OK;
}

oscar_status_t oscar_append_kv(const oscar_pool *pool, const oscar_bf16 *k_new, const oscar_bf16 *v_new,
                               oscar_stream_t stream) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  if (k_new == nullptr || v_new == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "k_new/v_new NULL");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 7u)
    return fail(OSCAR_ERR_INVALID_ARG, "k_new and v_new must be 8-byte aligned");
  if ((st = check_io(k_new, "k_new")) != OSCAR_OK || (st = check_io(v_new, "v_new")) != OSCAR_OK) return st;
  return cuda_status(launch_demote(a, nullptr, 2, k_new, v_new, static_cast<cudaStream_t>(stream)), "append_kv");
}

// Decode paths.  Whole-vector groups (128): the warp-MMA kernels of decode_v1.cu (uniform levels, or a
// codebook's indicator planes).  Groups of 32 or 64 with uniform levels: the tcgen05 kernels of decode_tc.cu
// (one accumulator column pair per group); with a codebook: the CUDA-core kernels of decode.cu.
// OSCAR_DECODE_TC=1 in the environment sends uniform pools of group size 128 to the tcgen05 kernels as well.
enum class Path { TC, V1, CORE };
static bool force_tc() {
  static const bool on = [] {
    const char *e = getenv("OSCAR_DECODE_TC");
    return e != nullptr && e[0] == '1' && e[1] == '\0';
  }();
  return on;
}
static Path decode_path(const PoolArgs &a) {
  const bool uniform = a.cb_k == nullptr && a.cb_v == nullptr;
  if (a.g == OSCAR_HEAD_DIM) return (uniform && force_tc()) ? Path::TC : Path::V1;
  return uniform ? Path::TC : Path::CORE;
}

// Workspace bytes a call needs at least (min) or the size that enables everything (the group-128 path's
// dynamic tail of the history split: oscar_decode_workspace_size reports it).
static size_t ws_min(const PoolArgs &a, int num_splits);
static size_t ws_need(const PoolArgs &a, int num_splits) {
  switch (decode_path(a)) {
    case Path::TC: return tc_ws_bytes(a);
    case Path::V1: return v1_ws_bytes(a, true);
    default: return decode_ws_bytes(a, num_splits == 0 ? auto_splits(a) : num_splits);
  }
}

static size_t ws_min(const PoolArgs &a, int num_splits) {
  return decode_path(a) == Path::V1 ? v1_ws_bytes(a, false) : ws_need(a, num_splits);
}

oscar_status_t oscar_decode_workspace_size(const oscar_pool *pool, int32_t num_splits, size_t *bytes) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  if (bytes == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "bytes is NULL");
  if (num_splits < 0) return fail(OSCAR_ERR_INVALID_ARG, "num_splits < 0");
  *bytes = ws_need(a, num_splits);
  return OSCAR_OK;
}

oscar_status_t oscar_decode_attention(const oscar_pool *pool, const oscar_bf16 *q, float *out, float softmax_scale,
                                      int32_t num_splits, void *ws, size_t ws_bytes, oscar_stream_t stream) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  if (q == nullptr || out == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "q/out NULL");
  if (!(softmax_scale > 0.0f)) return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be > 0");
  if (num_splits < 0) return fail(OSCAR_ERR_INVALID_ARG, "num_splits < 0");
  const Path path = decode_path(a);
  const size_t need = ws_min(a, num_splits);
  if (ws == nullptr || ws_bytes < need) return fail(OSCAR_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (path != Path::CORE && (reinterpret_cast<uintptr_t>(q) & 15u))
    return fail(OSCAR_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return fail(OSCAR_ERR_INVALID_ARG, "ws must be 16-byte aligned");
  if ((st = check_io(q, "q")) != OSCAR_OK || (st = check_io(out, "out")) != OSCAR_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  float *w = static_cast<float *>(ws);
  switch (path) {
    case Path::TC: return cuda_status(launch_decode_tc(a, q, out, softmax_scale, w, s), "decode_attention");
    case Path::V1:
      return cuda_status(launch_decode_v1(a, q, out, softmax_scale, w, s, ws_bytes >= v1_ws_bytes(a, true)),
                         "decode_attention");
    default:
      return cuda_status(launch_decode(a, q, out, softmax_scale, num_splits == 0 ? auto_splits(a) : num_splits, w, s),
                         "decode_attention");
  }
}

oscar_status_t oscar_decode_step(const oscar_pool *pool, const oscar_bf16 *k_new, const oscar_bf16 *v_new,
                                 const oscar_bf16 *q, float *out, float softmax_scale, void *ws, size_t ws_bytes,
                                 oscar_stream_t stream) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  if (k_new == nullptr || v_new == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "k_new/v_new NULL");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  if (q == nullptr || out == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "q/out NULL");
  if (!(softmax_scale > 0.0f)) return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be > 0");
  if ((st = check_io(k_new, "k_new")) != OSCAR_OK || (st = check_io(v_new, "v_new")) != OSCAR_OK ||
      (st = check_io(q, "q")) != OSCAR_OK || (st = check_io(out, "out")) != OSCAR_OK)
    return st;
  const Path path = decode_path(a);
  if (path == Path::CORE) {
    if ((st = oscar_append_kv(pool, k_new, v_new, stream)) != OSCAR_OK) return st;
    return oscar_decode_attention(pool, q, out, softmax_scale, 0, ws, ws_bytes, stream);
  }
  const size_t need = ws_min(a, 0);
  if (ws == nullptr || ws_bytes < need) return fail(OSCAR_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (reinterpret_cast<uintptr_t>(q) & 15u) return fail(OSCAR_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return fail(OSCAR_ERR_INVALID_ARG, "ws must be 16-byte aligned");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == Path::TC)
    return cuda_status(launch_decode_tc(a, q, out, softmax_scale, static_cast<float *>(ws), s, k_new, v_new),
                       "decode_step");
  return cuda_status(launch_step_v1(a, k_new, v_new, q, out, softmax_scale, static_cast<float *>(ws), s,
                                    ws_bytes >= v1_ws_bytes(a, true)),
                     "decode_step");
}

oscar_status_t oscar_bf16_prefill(const oscar_bf16_cache *cache, int32_t seq, int64_t len, const oscar_bf16 *k,
                                  const oscar_bf16 *v, oscar_stream_t stream) {
  CacheArgs a;
  oscar_status_t st = check_cache(cache, a);
  if (st != OSCAR_OK) return st;
  if (seq < 0 || seq >= a.B) return fail(OSCAR_ERR_INVALID_ARG, "seq %d outside [0, %d)", seq, a.B);
  if (len < 0 || len > (int64_t)a.max_pages * OSCAR_PAGE_TOKENS)
    return fail(OSCAR_ERR_INVALID_ARG, "len %lld outside [0, max_pages*64]", (long long)len);
  if (len > 0 && (k == nullptr || v == nullptr)) return fail(OSCAR_ERR_INVALID_ARG, "k/v NULL");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  return cuda_status(launch_bf16_prefill(a, seq, (int)len, k, v, static_cast<cudaStream_t>(stream)), "bf16_prefill");
}

oscar_status_t oscar_bf16_append_kv(const oscar_bf16_cache *cache, const oscar_bf16 *k_new, const oscar_bf16 *v_new,
                                    oscar_stream_t stream) {
  CacheArgs a;
  oscar_status_t st = check_cache(cache, a);
  if (st != OSCAR_OK) return st;
  if (k_new == nullptr || v_new == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "k_new/v_new NULL");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  return cuda_status(launch_bf16_append(a, k_new, v_new, static_cast<cudaStream_t>(stream)), "bf16_append_kv");
}

oscar_status_t oscar_bf16_decode_workspace_size(const oscar_bf16_cache *cache, size_t *bytes) {
  CacheArgs a;
  oscar_status_t st = check_cache(cache, a);
  if (st != OSCAR_OK) return st;
  if (bytes == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = bf16_ws_bytes(a);
  return OSCAR_OK;
}

static oscar_status_t bf16_decode(const oscar_bf16_cache *cache, const oscar_bf16 *k_new, const oscar_bf16 *v_new,
                                  const oscar_bf16 *q, float *out, float softmax_scale, void *ws, size_t ws_bytes,
                                  oscar_stream_t stream, const char *what) {
  CacheArgs a;
  oscar_status_t st = check_cache(cache, a);
  if (st != OSCAR_OK) return st;
  if (q == nullptr || out == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "q/out NULL");
  if ((reinterpret_cast<uintptr_t>(q) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u))
    return fail(OSCAR_ERR_INVALID_ARG, "q and out must be 4-byte aligned");
  if (!(softmax_scale > 0.0f)) return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be > 0");
  const size_t need = bf16_ws_bytes(a);
  if (ws == nullptr || ws_bytes < need) return fail(OSCAR_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  return cuda_status(launch_bf16_decode(a, q, out, softmax_scale, static_cast<float *>(ws),
                                        static_cast<cudaStream_t>(stream), k_new, v_new),
                     what);
}

oscar_status_t oscar_bf16_decode_attention(const oscar_bf16_cache *cache, const oscar_bf16 *q, float *out,
                                           float softmax_scale, void *ws, size_t ws_bytes, oscar_stream_t stream) {
  return bf16_decode(cache, nullptr, nullptr, q, out, softmax_scale, ws, ws_bytes, stream, "bf16_decode_attention");
}

oscar_status_t oscar_bf16_decode_step(const oscar_bf16_cache *cache, const oscar_bf16 *k_new,
                                      const oscar_bf16 *v_new, const oscar_bf16 *q, float *out,
                                      float softmax_scale, void *ws, size_t ws_bytes, oscar_stream_t stream) {
  if (k_new == nullptr || v_new == nullptr) return fail(OSCAR_ERR_INVALID_ARG, "k_new/v_new NULL");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return fail(OSCAR_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  return bf16_decode(cache, k_new, v_new, q, out, softmax_scale, ws, ws_bytes, stream, "bf16_decode_step");
}

}  // extern "C"

oscar_status_t oscar::decode_workspace_min(const oscar_pool *pool, size_t *bytes) {
  PoolArgs a;
  oscar_status_t st = check_pool(pool, a);
  if (st != OSCAR_OK) return st;
  *bytes = ws_min(a, 0);
  return OSCAR_OK;
}

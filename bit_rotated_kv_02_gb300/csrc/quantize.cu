// Demotion, append and prefill kernels of the three-segment pool.
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": a new token is
// first written into the recent window; as decoding advances the oldest recent token is rotated,
// clipped, quantized and packed by a fused kernel and demoted into the INT2 history; sink and
// recent stay BF16.
#include <algorithm>

#include "oscar_internal.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {

// ---------------------------------------------------------------------------------------------
// Demote (and optionally append): grid (2 * Hkv, B), 256 threads; CTA 2h handles the K vector and CTA
// 2h + 1 the V vector of KV head h of sequence blockIdx.y.  Each of the 8 warps holds 16 rows of R in
// registers (loaded at entry, with the appended token and the pool counters: a demotion is a chain of
// dependent reads, so everything independent is issued first); warp 0 combines the partial dots and
// quantizes.  Every CTA reads the sequence's counters before any CTA of that sequence can change them:
// the last CTA to arrive (arrival counter pool.sync[b]) updates the counters and returns the arrival
// counter to zero.
// mode 0: demote where recent_len == 256; mode 1: demote where mask[b] != 0 && recent_len > 0;
// mode 2: as mode 0, then append k_new/v_new.
constexpr int DEMOTE_WARPS = 8, DEMOTE_ROWS = D / DEMOTE_WARPS;  // 16 rows of R per warp
constexpr int RS_LD = D + 4;  // padded row stride of the shared copy of R (16-byte rows, 4-way reads)
constexpr size_t DEMOTE_SMEM = (size_t)D * RS_LD * sizeof(float);
__global__ void __launch_bounds__(256, 1) demote_append_kernel(PoolArgs p, const int32_t *mask, int mode,
                                                            const uint16_t *k_new, const uint16_t *v_new) {
  __shared__ float xs[D];
  __shared__ float pacc[DEMOTE_WARPS][32][4], psab[DEMOTE_WARPS][32][4];
  __shared__ int s_ok;
  __shared__ float qred[16];       // the quantizer's group extremes
  extern __shared__ float4 rs4[];  // this CTA's R, row stride RS_LD floats, for the Dot2 tier
  pdl_wait();
  pdl_trigger();
  const int kvh = blockIdx.x >> 1, kv = blockIdx.x & 1, b = blockIdx.y;  // kv 0 = K, 1 = V
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float *Rw = (kv == 0 ? p.R_k : p.R_v) + (size_t)kvh * D * D;
  float4 rrow[DEMOTE_ROWS];
  {
    const float4 *R4 = reinterpret_cast<const float4 *>(Rw) + (size_t)(DEMOTE_ROWS * warp) * (D / 4) + lane;
#pragma unroll
    for (int i = 0; i < DEMOTE_ROWS; ++i) rrow[i] = R4[i * (D / 4)];
#pragma unroll
    for (int i = 0; i < DEMOTE_ROWS; ++i) rs4[(DEMOTE_ROWS * warp + i) * (RS_LD / 4) + lane] = rrow[i];
  }
  // the appended token's row (mode 2; warp 0), also independent of the counters
  uint2 newrow = make_uint2(0u, 0u);
  if (mode == 2 && warp == 0)
    newrow = reinterpret_cast<const uint2 *>((kv == 0 ? k_new : v_new) + ((size_t)b * p.Hkv + kvh) * D)[lane];
  const int slen = p.sink_len[b], hl = p.hist_len[b], rs = p.recent_start[b], rl = p.recent_len[b];
  const bool counters_ok = slen >= 0 && slen <= SINK && hl >= 0 && rs >= 0 && rs < RECENT && rl >= 0 && rl <= RECENT;
  const bool want = counters_ok && ((mode == 1) ? (mask[b] != 0 && rl > 0) : (rl == RECENT));
  // the oldest recent vector and the page-table entry are read together
  uint2 xw = make_uint2(0u, 0u);
  if (want && warp == 0)
    xw = reinterpret_cast<const uint2 *>((kv == 0 ? p.recent_k : p.recent_v) +
                                         (((size_t)b * p.Hkv + kvh) * RECENT + rs) * D)[lane];
  bool demote = want;
  int page = -1;
  if (demote) {
    const int pidx = hl / PAGE;
    if (pidx >= p.max_pages) {
      demote = false;
      if (threadIdx.x == 0) atomicOr(p.err, OSCAR_DEVERR_HISTORY_FULL);
    } else {
      page = p.page_table[(size_t)b * p.max_pages + pidx];
      if (page < 0 || page >= p.num_pages) {
        demote = false;
        if (threadIdx.x == 0) atomicOr(p.err, OSCAR_DEVERR_PAGE_INDEX);
      }
    }
  }
  if (!counters_ok && threadIdx.x == 0) atomicOr(p.err, OSCAR_DEVERR_COUNTERS);
  // A demotion that cannot be stored leaves the whole sequence unchanged (no append either).
  const bool blocked = want && !demote;
  if (demote) {
    if (warp == 0) {
      xs[4 * lane + 0] = bf16_to_f32(xw.x & 0xffffu);
      xs[4 * lane + 1] = bf16_to_f32(xw.x >> 16);
      xs[4 * lane + 2] = bf16_to_f32(xw.y & 0xffffu);
      xs[4 * lane + 3] = bf16_to_f32(xw.y >> 16);
    }
    __syncthreads();
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, sab[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < DEMOTE_ROWS; ++i) {
      const float xi = xs[DEMOTE_ROWS * warp + i], ax = fabsf(xi);
      acc[0] = fmaf(xi, rrow[i].x, acc[0]);
      acc[1] = fmaf(xi, rrow[i].y, acc[1]);
      acc[2] = fmaf(xi, rrow[i].z, acc[2]);
      acc[3] = fmaf(xi, rrow[i].w, acc[3]);
      sab[0] = fmaf(ax, fabsf(rrow[i].x), sab[0]);
      sab[1] = fmaf(ax, fabsf(rrow[i].y), sab[1]);
      sab[2] = fmaf(ax, fabsf(rrow[i].z), sab[2]);
      sab[3] = fmaf(ax, fabsf(rrow[i].w), sab[3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) { pacc[warp][lane][k] = acc[k]; psab[warp][lane][k] = sab[k]; }
    __syncthreads();
    if (threadIdx.x < D) {  // thread e quantizes element e (the warps' partial sums in the order one warp adds them)
      const int k = threadIdx.x & 3, l = threadIdx.x >> 2;
      float a8 = 0.f, s8 = 0.f;
#pragma unroll
      for (int w = 0; w < DEMOTE_WARPS; ++w) { a8 += pacc[w][l][k]; s8 += psab[w][l][k]; }
      const float clip = (kv == 0 ? p.clip_k : p.clip_v)[kvh];
      const size_t row = ((size_t)page * p.Hkv + kvh) * PAGE + (hl % PAGE);
      QuantStats st{0, 0, 0};
      const float *cb = kv == 0 ? p.cb_k : p.cb_v;
      quantize_from_dots_cta(xs, Rw, reinterpret_cast<const float *>(rs4), RS_LD, a8, s8, clip, p.g,
                             (kv == 0 ? p.codes_k : p.codes_v) + row * (D / 4),
                             (kv == 0 ? p.scale_k : p.scale_v) + row * p.ng, (kv == 0 ? p.zero_k : p.zero_v) + row * p.ng,
                             st, cb != nullptr ? cb + 4 * kvh : nullptr, qred, 1);
    }
  }
  __syncthreads();  // the demoted slot is read before the append may overwrite it
  const bool append = mode == 2 && counters_ok && !blocked;
  int nslen = slen, nhl = hl, nrs = rs, nrl = rl;
  if (demote) { nhl = hl + 1; nrs = (rs + 1) % RECENT; nrl = rl - 1; }
  if (append && warp == 0) {
    uint16_t *dst;
    if (nslen < SINK && nhl == 0 && nrl == 0) {
      dst = (kv == 0 ? p.sink_k : p.sink_v) + (((size_t)b * p.Hkv + kvh) * SINK + nslen) * D;
    } else {
      dst = (kv == 0 ? p.recent_k : p.recent_v) + (((size_t)b * p.Hkv + kvh) * RECENT + (nrs + nrl) % RECENT) * D;
    }
    reinterpret_cast<uint2 *>(dst)[lane] = newrow;
  }
  if (append) {
    if (nslen < SINK && nhl == 0 && nrl == 0) nslen += 1;
    else nrl += 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int arrived = atomicAdd(p.sync + b, 1);
    s_ok = arrived == 2 * p.Hkv - 1;
  }
  __syncthreads();
  if (s_ok && threadIdx.x == 0) {
    __threadfence();
    if (counters_ok && !blocked) {
      p.sink_len[b] = nslen;
      p.hist_len[b] = nhl;
      p.recent_start[b] = nrs;
      p.recent_len[b] = nrl;
    }
    p.sync[b] = 0;
  }
}

// ---------------------------------------------------------------------------------------------
// Rotate / clip / quantize / pack with a codebook (the Lloyd-Max levels of this (KV head, K or V); the
// tensor-core bulk kernel serves the uniform levels): grid (ctas per head, Hkv), 256 threads.  The CTA
// holds R of its KV head in shared memory (padded rows); warp w quantizes rows r = 8 blockIdx.x + w,
// stepping by 8 gridDim.x: dots by FMA over the 128 rows of R (lane: 4 columns), then quantize_from_dots
// with the codebook, its compensated-dot tier reading the shared copy of R.  Output rows as in
// launch_quantize_rows (dense, or through the page table).
__global__ void __launch_bounds__(256, 1) quantize_rows_cb_kernel(int64_t n, int Hkv, int g, const uint16_t *x,
                                                                int64_t x_row_stride, const float *R32,
                                                                const float *clip, const float *cb, uint8_t *codes,
                                                                uint16_t *scale, uint16_t *zero, const int32_t *pt,
                                                                int num_pages, uint32_t *err, uint32_t *stats) {
  extern __shared__ float4 rs4[];  // R of this head, row stride RS_LD floats
  __shared__ float xs[DEMOTE_WARPS][D];
  const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float *Rw = R32 + (size_t)h * D * D;
  for (int i = threadIdx.x; i < D * (D / 4); i += blockDim.x)
    rs4[(i / (D / 4)) * (RS_LD / 4) + (i % (D / 4))] = reinterpret_cast<const float4 *>(Rw)[i];
  __syncthreads();
  const float *Rs = reinterpret_cast<const float *>(rs4);
  const float c = clip[h];
  const int ng = D / g;
  QuantStats st{0, 0, 0};
  for (int64_t r = (int64_t)blockIdx.x * DEMOTE_WARPS + warp; r < n; r += (int64_t)gridDim.x * DEMOTE_WARPS) {
    size_t drow;
    if (pt == nullptr) {
      drow = (size_t)r * Hkv + h;
    } else {
      const int page = pt[r / PAGE];
      if (page < 0 || page >= num_pages) {
        if (lane == 0 && err != nullptr) atomicOr(err, OSCAR_DEVERR_PAGE_INDEX);
        continue;
      }
      drow = ((size_t)page * Hkv + h) * PAGE + (size_t)(r % PAGE);
    }
    load_vec_to_smem(x + (size_t)r * x_row_stride + (size_t)h * D, xs[warp]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, sab[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int i = 0; i < D; ++i) {
      const float xi = xs[warp][i], ax = fabsf(xi);
      const float4 rv = rs4[i * (RS_LD / 4) + lane];
      acc[0] = fmaf(xi, rv.x, acc[0]); acc[1] = fmaf(xi, rv.y, acc[1]);
      acc[2] = fmaf(xi, rv.z, acc[2]); acc[3] = fmaf(xi, rv.w, acc[3]);
      sab[0] = fmaf(ax, fabsf(rv.x), sab[0]); sab[1] = fmaf(ax, fabsf(rv.y), sab[1]);
      sab[2] = fmaf(ax, fabsf(rv.z), sab[2]); sab[3] = fmaf(ax, fabsf(rv.w), sab[3]);
    }
    quantize_from_dots(xs[warp], Rw, Rs, RS_LD, acc, sab, c, g, codes + drow * (D / 4), scale + drow * ng,
                       zero + drow * ng, st, cb + 4 * h);
    __syncwarp();
  }
  flush_stats(stats, st);
}

// Copy token rows [t0, t0+n) of x [L][Hkv][D] into dst [Hkv][cap][D] rows [0, n) of one sequence.
__global__ void copy_rows_kernel(const uint16_t *x, int64_t t0, int n, int Hkv, uint16_t *dst, int cap) {
  const int kvh = blockIdx.y;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n * (D / 8); i += gridDim.x * blockDim.x) {
    const int t = i / (D / 8), c = i % (D / 8);
    reinterpret_cast<uint4 *>(dst + ((size_t)kvh * cap + t) * D)[c] =
        reinterpret_cast<const uint4 *>(x + ((size_t)(t0 + t) * Hkv + kvh) * D)[c];
  }
}

__global__ void set_counters_kernel(PoolArgs p, int b, int slen, int hl, int rl) {
  p.sink_len[b] = slen;
  p.hist_len[b] = hl;
  p.recent_start[b] = 0;
  p.recent_len[b] = rl;
}

// ---- launchers ------------------------------------------------------------------------------
cudaError_t launch_demote(const PoolArgs &p, const int32_t *mask, int mode, const uint16_t *k_new,
                          const uint16_t *v_new, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(demote_append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DEMOTE_SMEM);
  if (e != cudaSuccess) return e;
  profile_begin(OSCAR_PROFILE_DEMOTE, s);
  e = launch_pdl(demote_append_kernel, dim3(2 * p.Hkv, p.B), dim3(256), DEMOTE_SMEM, s, p, mask, mode, k_new, v_new);
  profile_end(OSCAR_PROFILE_DEMOTE, s);
  return e;
}

// skip: the first `skip` history pages are already in place (shared with another sequence's identical
// prefix through the page table) and are neither quantized nor written.
cudaError_t launch_quantize_rows_cb(int64_t n, int Hkv, int g, const uint16_t *x, int64_t x_row_stride,
                                    const float *R32, const float *clip, const float *cb, uint8_t *codes,
                                    uint16_t *scale, uint16_t *zero, const int32_t *pt, int num_pages, uint32_t *err,
                                    uint32_t *stats, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(quantize_rows_cb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)DEMOTE_SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n + DEMOTE_WARPS - 1) / DEMOTE_WARPS;
  const int per_head = (int)std::min<int64_t>(want, std::max(1, 2 * sms / Hkv));
  quantize_rows_cb_kernel<<<dim3(per_head, Hkv), 256, DEMOTE_SMEM, s>>>(n, Hkv, g, x, x_row_stride, R32, clip, cb,
                                                                       codes, scale, zero, pt, num_pages, err, stats);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PoolArgs &p, int b, int64_t L, const uint16_t *k, const uint16_t *v, uint32_t *stats,
                           cudaStream_t s, int skip) {
  const int ns = (int)(L < SINK ? L : SINK);
  const int64_t rest = L - ns;
  const int nr = (int)(rest < RECENT ? rest : RECENT);
  const int64_t nh = L - ns - nr;
  const int64_t stride = (int64_t)p.Hkv * D;
  cudaError_t e;
  if (ns > 0) {
    copy_rows_kernel<<<dim3(8, p.Hkv), 256, 0, s>>>(k, 0, ns, p.Hkv, p.sink_k + (size_t)b * p.Hkv * SINK * D, SINK);
    copy_rows_kernel<<<dim3(8, p.Hkv), 256, 0, s>>>(v, 0, ns, p.Hkv, p.sink_v + (size_t)b * p.Hkv * SINK * D, SINK);
  }
  if (nr > 0) {
    copy_rows_kernel<<<dim3(16, p.Hkv), 256, 0, s>>>(k, ns + nh, nr, p.Hkv,
                                                     p.recent_k + (size_t)b * p.Hkv * RECENT * D, RECENT);
    copy_rows_kernel<<<dim3(16, p.Hkv), 256, 0, s>>>(v, ns + nh, nr, p.Hkv,
                                                     p.recent_v + (size_t)b * p.Hkv * RECENT * D, RECENT);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t first = (int64_t)skip * PAGE;  // history rows [first, nh) are written
  if (nh > first) {
    const int32_t *pt = p.page_table + (size_t)b * p.max_pages + skip;
    const int64_t n = nh - first, x0 = (int64_t)ns + first;
    e = p.cb_k != nullptr
            ? launch_quantize_rows_cb(n, p.Hkv, p.g, k + (size_t)x0 * stride, stride, p.R_k, p.clip_k, p.cb_k,
                                      p.codes_k, p.scale_k, p.zero_k, pt, p.num_pages, p.err, stats, s)
            : launch_quantize_rows(n, p.Hkv, p.g, k + (size_t)x0 * stride, stride, p.R_k, p.clip_k, p.codes_k,
                                   p.scale_k, p.zero_k, pt, p.num_pages, p.err, stats, s);
    if (e != cudaSuccess) return e;
    e = p.cb_v != nullptr
            ? launch_quantize_rows_cb(n, p.Hkv, p.g, v + (size_t)x0 * stride, stride, p.R_v, p.clip_v, p.cb_v,
                                      p.codes_v, p.scale_v, p.zero_v, pt, p.num_pages, p.err, stats, s)
            : launch_quantize_rows(n, p.Hkv, p.g, v + (size_t)x0 * stride, stride, p.R_v, p.clip_v, p.codes_v,
                                   p.scale_v, p.zero_v, pt, p.num_pages, p.err, stats, s);
    if (e != cudaSuccess) return e;
  }
  set_counters_kernel<<<1, 1, 0, s>>>(p, b, ns, (int)nh, nr);
  return cudaGetLastError();
}

}  // namespace oscar

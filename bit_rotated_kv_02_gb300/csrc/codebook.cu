// Lloyd-Max codebook calibration: four dequantization levels per KV head in place of the uniform INT2
// levels 0, 1, 2, 3 ("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", the closing comparison with
// TurboQuant: the newest OSCAR code adds a Lloyd-Max codebook on top of the attention-aware rotation).
//
// A level lives in the group's own coordinate t = (x_rot - zero) / scale, with the scale and zero point
// of the uniform quantizer (so a code still dequantizes to zero + scale * l[code]).  Calibration:
//   1. calib_t_kernel: t of every element of the calibration rows (rotation by FMA dots with R in shared
//      memory, the group's clipped min/max, the bf16 scale and zero, one IEEE division); groups whose
//      scale is zero or not finite store NaN and take no part;
//   2. lloyd_kernel: one CTA per KV head runs Lloyd's method on its values from (0, 1, 2, 3): midpoints of
//      the levels, the cell of each value (nearest level, ties to the even code), the mean of each cell
//      (an empty cell keeps its level), until no level moves or the iteration limit.
// Cell sums are taken as deviations from the cell's current level (float32 within a thread, float64
// across threads, in a fixed order), so a converged assignment gives identical sums and the loop stops.
#include <cstdint>

#include "kernels.h"
#include "oscar_internal.cuh"

namespace oscar {
namespace {

constexpr int CAL_WARPS = 8;
constexpr int CAL_LD = D + 4;  // padded row stride of the shared copy of R
constexpr size_t CAL_SMEM = (size_t)D * CAL_LD * sizeof(float);
constexpr int LLOYD_THREADS = 1024;

// grid (ctas per head, Hkv), 256 threads; t [Hkv][n * D]: element (row r, channel j) at r * D + j.
__global__ void __launch_bounds__(256, 1) calib_t_kernel(int64_t n, int Hkv, int g, const uint16_t *x,
                                                        const float *R32, const float *clip, float *t) {
  extern __shared__ float4 rs4[];
  __shared__ float xs[CAL_WARPS][D];
  const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float4 *Rw = reinterpret_cast<const float4 *>(R32 + (size_t)h * D * D);
  for (int i = threadIdx.x; i < D * (D / 4); i += blockDim.x) rs4[(i / (D / 4)) * (CAL_LD / 4) + i % (D / 4)] = Rw[i];
  __syncthreads();
  const float c = clip[h];
  const int gl = g / 4;  // lanes per group
  float *th = t + (size_t)h * n * D;
  for (int64_t r = (int64_t)blockIdx.x * CAL_WARPS + warp; r < n; r += (int64_t)gridDim.x * CAL_WARPS) {
    load_vec_to_smem(x + ((size_t)r * Hkv + h) * D, xs[warp]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int i = 0; i < D; ++i) {
      const float xi = xs[warp][i];
      const float4 rv = rs4[i * (CAL_LD / 4) + lane];
      acc[0] = fmaf(xi, rv.x, acc[0]); acc[1] = fmaf(xi, rv.y, acc[1]);
      acc[2] = fmaf(xi, rv.z, acc[2]); acc[3] = fmaf(xi, rv.w, acc[3]);
    }
    float mn = fminf(fminf(acc[0], acc[1]), fminf(acc[2], acc[3]));
    float mx = fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3]));
    for (int off = gl / 2; off > 0; off >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(FULL, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
    }
    const float zf = bf16_to_f32(zero_of(c, mn)), sf = bf16_to_f32(scale_of(c, mn, mx));
    const bool valid = sf != 0.0f && isfinite(sf);
    float4 o;
    o.x = valid ? __fdiv_rn(__fsub_rn(acc[0], zf), sf) : __int_as_float(0x7fc00000);
    o.y = valid ? __fdiv_rn(__fsub_rn(acc[1], zf), sf) : __int_as_float(0x7fc00000);
    o.z = valid ? __fdiv_rn(__fsub_rn(acc[2], zf), sf) : __int_as_float(0x7fc00000);
    o.w = valid ? __fdiv_rn(__fsub_rn(acc[3], zf), sf) : __int_as_float(0x7fc00000);
    reinterpret_cast<float4 *>(th + (size_t)r * D)[lane] = o;
    __syncwarp();
  }
}

// grid Hkv, LLOYD_THREADS threads; cb_out [Hkv][4] float32.
__global__ void __launch_bounds__(LLOYD_THREADS, 1) lloyd_kernel(int64_t m, const float *t, int iters, float *cb_out) {
  __shared__ double red[LLOYD_THREADS / 32][8];
  __shared__ double lv[4];
  __shared__ int stop;
  const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float *th = t + (size_t)h * m;
  if (threadIdx.x < 4) lv[threadIdx.x] = (double)threadIdx.x;
  if (threadIdx.x == 0) stop = 0;
  __syncthreads();
  for (int it = 0; it < iters; ++it) {
    const double l0 = lv[0], l1 = lv[1], l2 = lv[2], l3 = lv[3];
    const double m0 = (l0 + l1) * 0.5, m1 = (l1 + l2) * 0.5, m2 = (l2 + l3) * 0.5;
    const float fl[4] = {(float)l0, (float)l1, (float)l2, (float)l3};
    float dev[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t cnt[4] = {0u, 0u, 0u, 0u};
    for (int64_t i = threadIdx.x; i < m; i += LLOYD_THREADS) {
      const float v = th[i];
      if (v != v) continue;  // group without a scale
      const double vd = (double)v;
      const int cell = (vd > m0) + (vd > m1) + (vd > m2) + (vd == m1);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (cell == k) { dev[k] += v - fl[k]; ++cnt[k]; }
    }
    // block reduction in a fixed order: warp shuffles, then warp 0 over the warps
    double s[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) { s[k] = (double)dev[k]; s[4 + k] = (double)cnt[k]; }
#pragma unroll
    for (int k = 0; k < 8; ++k)
      for (int off = 16; off > 0; off >>= 1) s[k] += __shfl_xor_sync(FULL, s[k], off);
    if (lane == 0)
#pragma unroll
      for (int k = 0; k < 8; ++k) red[warp][k] = s[k];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        double v = red[lane][k];
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(FULL, v, off);
        s[k] = v;
      }
      if (lane == 0) {
        double moved = 0.0;
        const double old[4] = {l0, l1, l2, l3};
        for (int k = 0; k < 4; ++k) {
          if (s[4 + k] > 0.0) {
            // the float32 level the deviations were taken from, plus their mean
            const double nl = (double)fl[k] + s[k] / s[4 + k];
            moved = fmax(moved, fabs(nl - old[k]));
            lv[k] = nl;
          }
        }
        if (moved <= 1e-12) stop = 1;
      }
    }
    __syncthreads();
    if (stop) break;
  }
  if (threadIdx.x < 4) cb_out[h * 4 + threadIdx.x] = (float)lv[threadIdx.x];
}

}  // namespace

size_t lloyd_ws_bytes(int64_t n, int Hkv) { return (size_t)n * Hkv * D * sizeof(float); }

cudaError_t launch_lloyd_max(int64_t n, int Hkv, int g, const uint16_t *x, const float *R32, const float *clip,
                             int iters, float *cb_out, void *ws, cudaStream_t s) {
  float *t = static_cast<float *>(ws);
  if (n > 0) {
    cudaError_t e = cudaFuncSetAttribute(calib_t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CAL_SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (n + CAL_WARPS - 1) / CAL_WARPS;
    const int per_head = (int)(want < (int64_t)(2 * sms / Hkv + 1) ? want : (int64_t)(2 * sms / Hkv + 1));
    calib_t_kernel<<<dim3(per_head, Hkv), 256, CAL_SMEM, s>>>(n, Hkv, g, x, R32, clip, t);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  lloyd_kernel<<<Hkv, LLOYD_THREADS, 0, s>>>(n * D, t, iters, cb_out);
  return cudaGetLastError();
}

}  // namespace oscar

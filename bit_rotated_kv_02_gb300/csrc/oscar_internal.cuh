// Internal device helpers of liboscar: bf16 storage, the INT2 quantizer arithmetic, and the
// warp-cooperative rotate -> clip -> quantize -> pack routine shared by demotion and prefill.
//
// Sources: "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计"
// (rotate, clip, quantize and pack the oldest recent token; 4 two-bit values per byte; scale and
// zero point).  The arithmetic below is this library's reading of those steps: x_hat is the float32
// nearest to the exact x · R; per group lo = c*min, hi = c*max, scale = bf16((hi-lo)/3),
// zero = bf16(lo), code = clamp(rint((x_hat - zero)/scale), 0, 3), all IEEE float32 round-to-nearest.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/oscar.h"

namespace oscar {

constexpr int D = OSCAR_HEAD_DIM;
constexpr int PAGE = OSCAR_PAGE_TOKENS;
constexpr int SINK = OSCAR_SINK_TOKENS;
constexpr int RECENT = OSCAR_RECENT_TOKENS;
constexpr unsigned FULL = 0xffffffffu;

// The pool passed by value to kernels.
struct PoolArgs {
  int B, Hq, Hkv, d, g, ng, num_pages, max_pages;
  uint16_t *sink_k, *sink_v, *recent_k, *recent_v;
  uint8_t *codes_k, *codes_v;
  uint16_t *scale_k, *zero_k, *scale_v, *zero_v;
  int32_t *page_table, *sink_len, *hist_len, *recent_start, *recent_len;
  const float *R_k, *R_v, *clip_k, *clip_v;
  uint32_t *err;
  int32_t *sync;
};

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// ---- quantizer arithmetic (explicit IEEE float32 round-to-nearest, no contraction) ----------
__device__ __forceinline__ uint16_t zero_of(float c, float mn) { return f32_to_bf16(__fmul_rn(c, mn)); }
__device__ __forceinline__ uint16_t scale_of(float c, float mn, float mx) {
  const float lo = __fmul_rn(c, mn), hi = __fmul_rn(c, mx);
  return f32_to_bf16(__fdiv_rn(__fsub_rn(hi, lo), 3.0f));
}
__device__ __forceinline__ int code_of(float x, float zero, float scale, bool valid) {
  if (!valid) return 0;
  const float t = __fdiv_rn(__fsub_rn(x, zero), scale);
  return (int)fminf(fmaxf(rintf(t), 0.0f), 3.0f);   // rintf: nearest, ties to even
}

// ---- exact rotated element --------------------------------------------------------------
// All 32 lanes cooperate on one element x_hat[j] = nearest float32 to sum_i x[i] * R[i][j].
// Products of a bf16 and a float32 are exact in float64; they are summed as a double-double
// (TwoSum error terms carried along), reduced with a butterfly that leaves every lane with the
// same value, and rounded to float32 by deciding the side of the float32 midpoint from the
// double-double's low part.  `unproven` is set when the result lies closer to a float32 midpoint
// than the double-double's error bound (~1e-27 of the sum of |products|).
__device__ __forceinline__ void two_sum(double a, double b, double &s, double &e) {
  s = a + b;
  const double bp = s - a;
  e = (a - (s - bp)) + (b - bp);
}

// Exact sign of (sum_i xs[i] * R[i][j]) - m, by fixed-point integer arithmetic: every product of a
// float32-held bf16 and a float32 is an integer (< 2^48) times a power of two, and m (a float32
// midpoint held in a double) is an integer < 2^53 times a power of two; all are aligned to the
// smallest exponent and summed in 128-bit integers.  Returns -1, 0 or +1, or 2 when the exponent
// span does not fit in 128 bits.  Runs serially on the calling lane (used only for exact ties).
// XF: callable giving x_i (a float32-held bf16) for i in [0, 128).
template <class XF>
__device__ inline int exact_sign_minus_f(XF xs, const float *R, int j, double m) {
  int emin = 0x7fffffff, etop = -0x7fffffff;
  for (int i = 0; i < D; ++i) {
    const float x = xs(i), r = R[i * D + j];
    if (x == 0.0f || r == 0.0f) continue;
    int ex, er;
    frexpf(x, &ex);
    frexpf(r, &er);
    const int e = ex + er - 48;            // product = (mx * mr) * 2^e with |mx|, |mr| < 2^24
    emin = min(emin, e);
    etop = max(etop, e + 48);
  }
  int em = 0;
  if (m != 0.0) {
    frexp(m, &em);
    emin = min(emin, em - 53);
    etop = max(etop, em);
  }
  if (emin == 0x7fffffff) return 0;        // every term is zero and m == 0
  if (etop - emin > 118) return 2;         // 7 bits of headroom for 128 terms + sign
  __int128 acc = 0;
  for (int i = 0; i < D; ++i) {
    const float x = xs(i), r = R[i * D + j];
    if (x == 0.0f || r == 0.0f) continue;
    int ex, er;
    const long long mx = (long long)ldexpf(frexpf(x, &ex), 24);
    const long long mr = (long long)ldexpf(frexpf(r, &er), 24);
    acc += (__int128)(mx * mr) << (ex + er - 48 - emin);
  }
  if (m != 0.0) acc -= (__int128)(long long)ldexp(frexp(m, &em), 53) << (em - 53 - emin);
  return acc > 0 ? 1 : (acc < 0 ? -1 : 0);
}

__device__ inline int exact_sign_minus(const float *xs, const float *R, int j, double m) {
  return exact_sign_minus_f([xs](int i) { return xs[i]; }, R, j, m);
}

template <class XF>
__device__ inline float exact_rot_elem_f(XF xs, const float *R, int j, bool &unproven) {
  const int lane = threadIdx.x & 31;
  double s = 0.0, c = 0.0, sa = 0.0;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    const int i = lane + 32 * k;
    const double p = (double)xs(i) * (double)R[i * D + j];
    double t, e;
    two_sum(s, p, t, e);
    s = t;
    c += e;
    sa += fabs(p);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double s2 = __shfl_xor_sync(FULL, s, off);
    const double c2 = __shfl_xor_sync(FULL, c, off);
    const double a2 = __shfl_xor_sync(FULL, sa, off);
    double t, e;
    two_sum(s, s2, t, e);
    s = t;
    c = (c + c2) + e;
    sa += a2;
  }
  double hi, lo;
  two_sum(s, c, hi, lo);
  const float rd = __double2float_rd(hi), ru = __double2float_ru(hi);
  if (rd == ru) return rd;                       // hi is a float32: |lo| < ulp64(hi)/2 cannot move it
  const double mid = 0.5 * ((double)rd + (double)ru);
  double dist = (hi - mid) + lo;                 // hi - mid is exact (Sterbenz)
  if (fabs(dist) <= 1e-27 * sa) {
    // Within the double-double's error bound of the midpoint (in practice an exact tie, which
    // bf16 x float32 products make possible): decide with exact integer arithmetic.
    int sg = 0;
    if ((threadIdx.x & 31) == 0) sg = exact_sign_minus_f(xs, R, j, mid);
    sg = __shfl_sync(FULL, sg, 0);
    if (sg == 2) unproven = true;
    else dist = (double)sg;
  }
  if (dist > 0.0) return ru;
  if (dist < 0.0) return rd;
  return __double2float_rn(hi);                  // exact tie: to even
}

__device__ inline float exact_rot_elem(const float *xs, const float *R, int j, bool &unproven) {
  return exact_rot_elem_f([xs](int i) { return xs[i]; }, R, j, unproven);
}

// ---- warp-cooperative rotate -> clip -> quantize -> pack of one head vector ----------------
// xs: this warp's float32 copy of the bf16 input vector (128 entries, shared memory).
// R:  row-major fp32 [128][128] (global or shared).  Lane l owns rotated channels 4l..4l+3.
// Fast path: sequential float32 FMA dots plus the running sum of |x_i R_ij|; the classical bound
// |fl(dot) - dot| <= gamma_128 * sum|x_i R_ij| (gamma_n = n u / (1 - n u), u = 2^-24) gives an
// interval [a, b] that must contain the correctly rounded x_hat.  scale/zero are taken from the
// interval when every corner gives the same bf16 result, and a code when both ends give the same
// code (every quantizer step is monotone); otherwise the affected elements are evaluated exactly.
struct QuantStats {
  uint32_t exact_elems, exact_groups, unproven;
};

// Partial fast-path dots over rows [i0, i1) of R: lane l accumulates channels 4l..4l+3 of x·R and of
// |x|·|R| (the latter bounds the rounding error of the former).
__device__ __forceinline__ void rot_dot_rows(const float *xs, const float *R, int i0, int i1, float (&acc)[4],
                                             float (&sab)[4]) {
  const int lane = threadIdx.x & 31;
  const float4 *R4 = reinterpret_cast<const float4 *>(R);
#pragma unroll 8
  for (int i = i0; i < i1; ++i) {
    const float xi = xs[i];
    const float ax = fabsf(xi);
    const float4 r = R4[i * (D / 4) + lane];
    acc[0] = fmaf(xi, r.x, acc[0]);
    acc[1] = fmaf(xi, r.y, acc[1]);
    acc[2] = fmaf(xi, r.z, acc[2]);
    acc[3] = fmaf(xi, r.w, acc[3]);
    sab[0] = fmaf(ax, fabsf(r.x), sab[0]);
    sab[1] = fmaf(ax, fabsf(r.y), sab[1]);
    sab[2] = fmaf(ax, fabsf(r.z), sab[2]);
    sab[3] = fmaf(ax, fabsf(r.w), sab[3]);
  }
}

// The same over exactly 32 rows starting at i0, with all 32 row loads issued before any use.
__device__ __forceinline__ void rot_dot_32rows(const float *xs, const float *R, int i0, float (&acc)[4],
                                               float (&sab)[4]) {
  const int lane = threadIdx.x & 31;
  const float4 *R4 = reinterpret_cast<const float4 *>(R) + (size_t)i0 * (D / 4) + lane;
  float4 r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = R4[i * (D / 4)];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float xi = xs[i0 + i], ax = fabsf(xi);
    acc[0] = fmaf(xi, r[i].x, acc[0]);
    acc[1] = fmaf(xi, r[i].y, acc[1]);
    acc[2] = fmaf(xi, r[i].z, acc[2]);
    acc[3] = fmaf(xi, r[i].w, acc[3]);
    sab[0] = fmaf(ax, fabsf(r[i].x), sab[0]);
    sab[1] = fmaf(ax, fabsf(r[i].y), sab[1]);
    sab[2] = fmaf(ax, fabsf(r[i].z), sab[2]);
    sab[3] = fmaf(ax, fabsf(r[i].w), sab[3]);
  }
}

// Quantize one vector from its fast-path dots (acc) and |x|·|R| sums (sab), however the 128
// products were grouped and ordered (the error bound below holds for any summation order).
__device__ inline void quantize_from_dots(const float *xs, const float *R, const float (&acc)[4], const float (&sab)[4],
                                          float clip, int g, uint8_t *codes_out, uint16_t *scale_out,
                                          uint16_t *zero_out, QuantStats &st) {
  const int lane = threadIdx.x & 31;
  // gamma_128 = 7.6294e-6; 8e-6 also covers the rounding of sab itself; 1e-37 covers underflow.
  float a[4], b[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float E = __fadd_ru(__fmul_ru(sab[k], 8.0e-6f), 1e-37f);
    a[k] = __fsub_rd(acc[k], E);
    b[k] = __fadd_ru(acc[k], E);
  }
  const int gl = g / 4;  // lanes per group (8, 16 or 32)
  float mn_lo = fminf(fminf(a[0], a[1]), fminf(a[2], a[3]));
  float mn_hi = fminf(fminf(b[0], b[1]), fminf(b[2], b[3]));
  float mx_lo = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
  float mx_hi = fmaxf(fmaxf(b[0], b[1]), fmaxf(b[2], b[3]));
  for (int off = gl / 2; off > 0; off >>= 1) {
    mn_lo = fminf(mn_lo, __shfl_xor_sync(FULL, mn_lo, off));
    mn_hi = fminf(mn_hi, __shfl_xor_sync(FULL, mn_hi, off));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(FULL, mx_lo, off));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(FULL, mx_hi, off));
  }
  uint16_t z = zero_of(clip, mn_lo);
  uint16_t s = scale_of(clip, mn_lo, mx_lo);
  const bool decided = z == zero_of(clip, mn_hi) && s == scale_of(clip, mn_lo, mx_hi) &&
                       s == scale_of(clip, mn_hi, mx_lo) && s == scale_of(clip, mn_hi, mx_hi);

  float xe[4];
  bool known[4] = {false, false, false, false};
  bool unproven = false;
  // Exact min/max where the interval leaves scale or zero open: only elements whose interval
  // reaches the group's extreme can be the extreme.
  bool candmin[4], candmax[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    candmin[k] = !decided && a[k] <= mn_hi;
    candmax[k] = !decided && b[k] >= mx_lo;
  }
  unsigned pend = __ballot_sync(FULL, candmin[0] || candmin[1] || candmin[2] || candmin[3] ||
                                          candmax[0] || candmax[1] || candmax[2] || candmax[3]);
  while (pend) {
    const int src = __ffs(pend) - 1;
    uint32_t mymask = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if ((candmin[k] || candmax[k]) && !known[k]) mymask |= 1u << k;
    mymask = __shfl_sync(FULL, mymask, src);
    const int k = __ffs(mymask) - 1;
    const float v = exact_rot_elem(xs, R, 4 * src + k, unproven);
    if (lane == src) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        if (kk == k) { xe[kk] = v; known[kk] = true; }
    }
    ++st.exact_elems;
    bool more = false;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) more |= (candmin[kk] || candmax[kk]) && !known[kk];
    pend = __ballot_sync(FULL, more);
  }
  {
    // every lane takes part in the reduction; only undecided groups use its result
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (candmin[k]) mn = fminf(mn, xe[k]);
      if (candmax[k]) mx = fmaxf(mx, xe[k]);
    }
    for (int off = gl / 2; off > 0; off >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(FULL, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
    }
    if (!decided) {
      z = zero_of(clip, mn);
      s = scale_of(clip, mn, mx);
    }
    st.exact_groups += __popc(__ballot_sync(FULL, !decided && (lane & (gl - 1)) == 0));
  }
  const float zf = bf16_to_f32(z), sf = bf16_to_f32(s);
  const bool valid = sf != 0.0f && isfinite(sf);
  int code[4];
  bool need[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (known[k]) {
      code[k] = code_of(xe[k], zf, sf, valid);
      need[k] = false;
    } else {
      code[k] = code_of(a[k], zf, sf, valid);
      need[k] = code[k] != code_of(b[k], zf, sf, valid);
    }
  }
  pend = __ballot_sync(FULL, need[0] || need[1] || need[2] || need[3]);
  while (pend) {
    const int src = __ffs(pend) - 1;
    uint32_t mymask = (need[0] ? 1u : 0u) | (need[1] ? 2u : 0u) | (need[2] ? 4u : 0u) | (need[3] ? 8u : 0u);
    mymask = __shfl_sync(FULL, mymask, src);
    const int k = __ffs(mymask) - 1;
    const float v = exact_rot_elem(xs, R, 4 * src + k, unproven);
    if (lane == src) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        if (kk == k) { code[kk] = code_of(v, zf, sf, valid); need[kk] = false; }
    }
    ++st.exact_elems;
    pend = __ballot_sync(FULL, need[0] || need[1] || need[2] || need[3]);
  }
  if (__any_sync(FULL, unproven) && lane == 0) ++st.unproven;
  codes_out[lane] = (uint8_t)(code[0] | (code[1] << 2) | (code[2] << 4) | (code[3] << 6));
  if ((lane & (gl - 1)) == 0) {
    scale_out[lane / gl] = s;
    zero_out[lane / gl] = z;
  }
}

__device__ inline void rotate_quantize_warp(const float *xs, const float *R, float clip, int g,
                                            uint8_t *codes_out, uint16_t *scale_out, uint16_t *zero_out,
                                            QuantStats &st) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, sab[4] = {0.f, 0.f, 0.f, 0.f};
  rot_dot_rows(xs, R, 0, D, acc, sab);
  quantize_from_dots(xs, R, acc, sab, clip, g, codes_out, scale_out, zero_out, st);
}

// Load one bf16 head vector (128 values, 8-byte aligned) into the warp's shared float32 buffer.
__device__ __forceinline__ void load_vec_to_smem(const uint16_t *x, float *xs) {
  const int lane = threadIdx.x & 31;
  const uint2 w = reinterpret_cast<const uint2 *>(x)[lane];
  xs[4 * lane + 0] = bf16_to_f32(w.x & 0xffffu);
  xs[4 * lane + 1] = bf16_to_f32(w.x >> 16);
  xs[4 * lane + 2] = bf16_to_f32(w.y & 0xffffu);
  xs[4 * lane + 3] = bf16_to_f32(w.y >> 16);
  __syncwarp();
}

__device__ __forceinline__ void flush_stats(uint32_t *stats, const QuantStats &st) {
  if (stats != nullptr && (threadIdx.x & 31) == 0) {
    if (st.exact_elems) atomicAdd(stats + 0, st.exact_elems);
    if (st.exact_groups) atomicAdd(stats + 1, st.exact_groups);
    if (st.unproven) atomicAdd(stats + 2, st.unproven);
  }
}

}  // namespace oscar

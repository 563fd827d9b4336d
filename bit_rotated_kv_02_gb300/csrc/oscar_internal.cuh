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
  const float *cb_k, *cb_v;  // [Hkv][4] codebook levels, or nullptr for the uniform levels 0, 1, 2, 3
};

// Device-side bounds checks of the debug build (compiled with -DOSCAR_DEBUG into liboscar_debug.so): a failed
// check ORs OSCAR_DEVERR_DEBUG_CHECK into the error word and the caller skips the access; the release build
// compiles them away.  They never trap: the context stays usable and the host reads the error word.
#ifdef OSCAR_DEBUG
#define OSCAR_DCHECK(cond, errp) ((cond) ? true : (atomicOr((errp), OSCAR_DEVERR_DEBUG_CHECK), false))
#else
#define OSCAR_DCHECK(cond, errp) true
#endif

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

// Codebook quantizer: the level l_i nearest to t = (x - zero) / scale, ties to the even index, from the
// float32 midpoints m = (m_0, m_1, m_2), m_i = (l_i + l_{i+1}) / 2: code = #{i : t > m_i} + (t == m_1).
// The uniform levels (0, 1, 2, 3) give clamp(rint(t), 0, 3).  Monotone in x for scale > 0.
__device__ __forceinline__ float3 level_midpoints(const float *cb) {
  return make_float3(__fmul_rn(__fadd_rn(cb[0], cb[1]), 0.5f), __fmul_rn(__fadd_rn(cb[1], cb[2]), 0.5f),
                     __fmul_rn(__fadd_rn(cb[2], cb[3]), 0.5f));
}
__device__ __forceinline__ int code_of_levels(float x, float zero, float scale, bool valid, float3 m) {
  if (!valid) return 0;
  const float t = __fdiv_rn(__fsub_rn(x, zero), scale);
  return (t > m.x) + (t > m.y) + (t > m.z) + (t == m.y);
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
// Fast path: float32 FMA dots plus the running sum of |x_i R_ij|; the classical bound
// |fl(dot) - dot| <= gamma_128 * sum|x_i R_ij| (gamma_n = n u / (1 - n u), u = 2^-24) gives an
// interval that must contain the correctly rounded x_hat.  Every quantizer step is monotone, so a
// decision taken at both ends of an interval holds for every value inside it.
struct QuantStats {
  uint32_t exact_elems, exact_groups, unproven;
};

// The same over 32 rows i0 .. i0+31 already in registers (r[i] = row i0 + i, this lane's four channels).
__device__ __forceinline__ void rot_dot_32rows_pre(const float *xs, const float4 (&r)[32], int i0, float (&acc)[4],
                                                   float (&sab)[4]) {
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

// Warp-cooperative interval [x, y] containing the float32 nearest to the exact x . R_j (xs: float32
// copy of the bf16 vector; R row-major fp32 with leading dimension ld, e.g. a padded shared copy).  Products are split error-free (p + e = x r, FMA),
// partial sums carry their rounding errors (TwoSum), and the errors are summed in plain float32,
// whose own error is below gamma_2n * gamma_n * sum|x r| < 2^-33 sum|x r|; the interval uses 2^-31
// times the computed sum.  Every lane returns the same interval.
__device__ __forceinline__ void two_sum_f32(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}
static __device__ __noinline__ float2 dot2_interval_xs(const float *xs, const float *R, int ld, int j) {
  const int lane = threadIdx.x & 31;
  float s = 0.f, c = 0.f, sab = 0.f;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    const int i = lane + 32 * k;
    const float xv = xs[i], rv = R[i * ld + j];
    const float p = __fmul_rn(xv, rv);
    const float e = fmaf(xv, rv, -p);
    float t, q;
    two_sum_f32(s, p, t, q);
    s = t;
    c = __fadd_rn(c, __fadd_rn(q, e));
    sab = fmaf(fabsf(xv), fabsf(rv), sab);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float s2 = __shfl_xor_sync(FULL, s, off);
    const float c2 = __shfl_xor_sync(FULL, c, off);
    const float a2 = __shfl_xor_sync(FULL, sab, off);
    float t, q;
    two_sum_f32(s, s2, t, q);
    s = t;
    c = __fadd_rn(__fadd_rn(c, c2), q);
    sab = __fadd_rn(sab, a2);
  }
  float hi, lo;
  two_sum_f32(s, c, hi, lo);
  const float B = __fadd_ru(__fmul_ru(sab, 0x1p-31f), 1e-36f);
  return make_float2(__fadd_rd(hi, __fsub_rd(lo, B)), __fadd_ru(hi, __fadd_ru(lo, B)));
}

// Quantize one vector from its fast-path dots (acc) and |x|·|R| sums (sab), however the 128
// products were grouped and ordered (the error bound below holds for any summation order).
// Every element carries an interval [lo, hi] that contains its correctly rounded x_hat: first the
// fast one; for the elements a decision needs, a Dot2 interval; if that still leaves the decision
// open, the exact value.  A group's zero is decided when both ends of its minimum's interval give
// the same bf16 zero, its scale when both extreme corners give the same bf16 scale (zero increases
// with the minimum; scale increases with the maximum and decreases with the minimum), and a code
// when both ends of the element's interval give the same code.
// R: the rotation in global memory (float64 / integer tier); R2, ld2: the same values for the Dot2
// tier (a shared-memory copy with row stride ld2, or R itself with ld2 = 128).
// cb: the four codebook levels of this (KV head, K/V), or nullptr for the uniform levels.
__device__ inline void quantize_from_dots(const float *xs, const float *R, const float *R2, int ld2,
                                          const float (&acc)[4], const float (&sab)[4], float clip, int g,
                                          uint8_t *codes_out, uint16_t *scale_out, uint16_t *zero_out,
                                          QuantStats &st, const float *cb = nullptr) {
  const int lane = threadIdx.x & 31;
  const int gl = g / 4;  // lanes per group (8, 16 or 32)
  // gamma_128 = 7.6294e-6; 8e-6 also covers the rounding of sab itself; 1e-37 covers underflow.
  float lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float E = __fadd_ru(__fmul_ru(sab[k], 8.0e-6f), 1e-37f);
    lo[k] = __fsub_rd(acc[k], E);
    hi[k] = __fadd_ru(acc[k], E);
  }
  auto group_min = [&](float v) {
    for (int off = gl / 2; off > 0; off >>= 1) v = fminf(v, __shfl_xor_sync(FULL, v, off));
    return v;
  };
  auto group_max = [&](float v) {
    for (int off = gl / 2; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, off));
    return v;
  };
  const float mn_lo = group_min(fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3])));
  const float mn_hi = group_min(fminf(fminf(hi[0], hi[1]), fminf(hi[2], hi[3])));
  const float mx_lo = group_max(fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3])));
  const float mx_hi = group_max(fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3])));
  uint16_t z = zero_of(clip, mn_lo), s = scale_of(clip, mn_hi, mx_lo);
  bool uz = z != zero_of(clip, mn_hi), us = s != scale_of(clip, mn_lo, mx_hi);
  st.exact_groups += __popc(__ballot_sync(FULL, (uz || us) && (lane & (gl - 1)) == 0));
  bool unproven = false;
  // candidates for the extremes: only elements whose interval reaches the group's extreme
  bool cmin[4], cmax[4], cand[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    cmin[k] = (uz || us) && lo[k] <= mn_hi;
    cmax[k] = us && hi[k] >= mx_lo;
    cand[k] = cmin[k] || cmax[k];
  }
  int done[4] = {-1, -1, -1, -1};  // highest tier already applied to the element
  // evaluate the flagged elements of the warp at `tier` (0: Dot2 interval, 1: exact value)
  auto evaluate = [&](const bool (&flag)[4], int tier) {
    uint32_t mine = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (flag[k] && done[k] < tier) mine |= 1u << k;
    while (__any_sync(FULL, mine != 0)) {
      const int src = __ffs(__ballot_sync(FULL, mine != 0)) - 1;
      const int k = __ffs(__shfl_sync(FULL, mine, src)) - 1;
      float2 iv;
      if (tier == 0) iv = dot2_interval_xs(xs, R2, ld2, 4 * src + k);
      else iv.x = iv.y = exact_rot_elem(xs, R, 4 * src + k, unproven);
      if (lane == src) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (kk == k) { lo[kk] = iv.x; hi[kk] = iv.y; done[kk] = tier; }
        mine &= mine - 1;
      }
      ++st.exact_elems;
    }
  };
  for (int tier = 0; tier < 2 && __any_sync(FULL, uz || us); ++tier) {
    evaluate(cand, tier);
    float a0 = INFINITY, a1 = INFINITY, b0 = -INFINITY, b1 = -INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (cmin[k]) { a0 = fminf(a0, lo[k]); a1 = fminf(a1, hi[k]); }
      if (cmax[k]) { b0 = fmaxf(b0, lo[k]); b1 = fmaxf(b1, hi[k]); }
    }
    a0 = group_min(a0);
    a1 = group_min(a1);
    b0 = group_max(b0);
    b1 = group_max(b1);
    if (uz) {
      const uint16_t z1 = zero_of(clip, a0);
      if (z1 == zero_of(clip, a1) || tier == 1) { z = z1; uz = false; }
    }
    if (us) {
      const uint16_t s1 = scale_of(clip, a1, b0);
      if (s1 == scale_of(clip, a0, b1) || tier == 1) { s = s1; us = false; }
    }
  }
  const float zf = bf16_to_f32(z), sf = bf16_to_f32(s);
  const bool valid = sf != 0.0f && isfinite(sf);
  const float3 mids = cb != nullptr ? level_midpoints(cb) : make_float3(0.f, 0.f, 0.f);
  auto code_at = [&](float x) { return cb != nullptr ? code_of_levels(x, zf, sf, valid, mids) : code_of(x, zf, sf, valid); };
  int code[4];
  for (int tier = 0; tier < 3; ++tier) {
    bool need[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      code[k] = code_at(lo[k]);
      need[k] = code[k] != code_at(hi[k]);
    }
    if (tier == 2 || !__any_sync(FULL, need[0] || need[1] || need[2] || need[3])) break;
    evaluate(need, tier);
  }
  if (__any_sync(FULL, unproven) && lane == 0) ++st.unproven;
  codes_out[lane] = (uint8_t)(code[0] | (code[1] << 2) | (code[2] << 4) | (code[3] << 6));
  if ((lane & (gl - 1)) == 0) {
    scale_out[lane / gl] = s;
    zero_out[lane / gl] = z;
  }
}

// Named barrier `bar` over 128 threads, and the OR of a predicate over them.
__device__ __forceinline__ void bar_sync128(int bar) { asm volatile("bar.sync %0, 128;\n" ::"r"(bar) : "memory"); }
__device__ __forceinline__ bool bar_or128(int bar, bool v) {
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
               : "=r"(r)
               : "r"((uint32_t)v), "r"(bar)
               : "memory");
  return r != 0;
}

// quantize_from_dots on the first 128 threads of a CTA (four warps, named barrier `bar`), one element per
// thread (element e = thread e): the same intervals, decisions and results, with a chain a quarter as long.
// A group's extremes combine its warps through `red` (shared memory, 16 floats); the Dot2 and exact
// evaluations run warp by warp over each warp's own flagged elements.
__device__ inline void quantize_from_dots_cta(const float *xs, const float *R, const float *R2, int ld2, float acc,
                                              float sab, float clip, int g, uint8_t *codes_out, uint16_t *scale_out,
                                              uint16_t *zero_out, QuantStats &st, const float *cb, float *red, int bar) {
  const int e = threadIdx.x & 127, lane = e & 31, warp = e >> 5;
  const int wpg = g / 32;              // warps per group (1, 2 or 4)
  const int gw0 = (warp / wpg) * wpg;  // the first warp of this thread's group
  // gamma_128 = 7.6294e-6; 8e-6 also covers the rounding of sab itself; 1e-37 covers underflow.
  const float E = __fadd_ru(__fmul_ru(sab, 8.0e-6f), 1e-37f);
  float lo = __fsub_rd(acc, E), hi = __fadd_ru(acc, E);
  // minima of a, b and maxima of c, d over the group
  auto group4 = [&](float &a, float &b, float &c, float &d) {
    for (int off = 16; off > 0; off >>= 1) {
      a = fminf(a, __shfl_xor_sync(FULL, a, off));
      b = fminf(b, __shfl_xor_sync(FULL, b, off));
      c = fmaxf(c, __shfl_xor_sync(FULL, c, off));
      d = fmaxf(d, __shfl_xor_sync(FULL, d, off));
    }
    if (wpg > 1) {
      bar_sync128(bar);  // every earlier read of red is done
      if (lane == 0) {
        red[4 * warp + 0] = a; red[4 * warp + 1] = b; red[4 * warp + 2] = c; red[4 * warp + 3] = d;
      }
      bar_sync128(bar);
      for (int w = gw0; w < gw0 + wpg; ++w) {
        a = fminf(a, red[4 * w + 0]); b = fminf(b, red[4 * w + 1]);
        c = fmaxf(c, red[4 * w + 2]); d = fmaxf(d, red[4 * w + 3]);
      }
    }
  };
  float mn_lo = lo, mn_hi = hi, mx_lo = lo, mx_hi = hi;
  group4(mn_lo, mn_hi, mx_lo, mx_hi);
  uint16_t z = zero_of(clip, mn_lo), s = scale_of(clip, mn_hi, mx_lo);
  bool uz = z != zero_of(clip, mn_hi), us = s != scale_of(clip, mn_lo, mx_hi);
  if ((uz || us) && (e & (g - 1)) == 0) ++st.exact_groups;
  bool unproven = false;
  // candidates for the extremes: only elements whose interval reaches the group's extreme
  const bool cmin = (uz || us) && lo <= mn_hi, cmax = us && hi >= mx_lo, cand = cmin || cmax;
  int done = -1;  // highest tier already applied to the element
  auto evaluate = [&](bool flag, int tier) {
    uint32_t mine = __ballot_sync(FULL, flag && done < tier);
    while (mine != 0) {
      const int src = __ffs(mine) - 1;
      mine &= mine - 1;
      float2 iv;
      if (tier == 0) iv = dot2_interval_xs(xs, R2, ld2, 32 * warp + src);
      else iv.x = iv.y = exact_rot_elem(xs, R, 32 * warp + src, unproven);
      if (lane == src) { lo = iv.x; hi = iv.y; done = tier; }
      ++st.exact_elems;
    }
  };
  for (int tier = 0; tier < 2; ++tier) {
    if (!bar_or128(bar, uz || us)) break;
    evaluate(cand, tier);
    float a0 = cmin ? lo : INFINITY, a1 = cmin ? hi : INFINITY, b0 = cmax ? lo : -INFINITY, b1 = cmax ? hi : -INFINITY;
    group4(a0, a1, b0, b1);
    if (uz) {
      const uint16_t z1 = zero_of(clip, a0);
      if (z1 == zero_of(clip, a1) || tier == 1) { z = z1; uz = false; }
    }
    if (us) {
      const uint16_t s1 = scale_of(clip, a1, b0);
      if (s1 == scale_of(clip, a0, b1) || tier == 1) { s = s1; us = false; }
    }
  }
  const float zf = bf16_to_f32(z), sf = bf16_to_f32(s);
  const bool valid = sf != 0.0f && isfinite(sf);
  const float3 mids = cb != nullptr ? level_midpoints(cb) : make_float3(0.f, 0.f, 0.f);
  auto code_at = [&](float x) { return cb != nullptr ? code_of_levels(x, zf, sf, valid, mids) : code_of(x, zf, sf, valid); };
  int code = 0;
  for (int tier = 0; tier < 3; ++tier) {
    code = code_at(lo);
    const bool need = code != code_at(hi);
    if (tier == 2 || !__any_sync(FULL, need)) break;
    evaluate(need, tier);
  }
  if (__any_sync(FULL, unproven) && lane == 0) ++st.unproven;
  const int c1 = __shfl_down_sync(FULL, code, 1), c2 = __shfl_down_sync(FULL, code, 2),
            c3 = __shfl_down_sync(FULL, code, 3);
  if ((lane & 3) == 0) codes_out[e >> 2] = (uint8_t)(code | (c1 << 2) | (c2 << 4) | (c3 << 6));
  if ((e & (g - 1)) == 0) {
    scale_out[e / g] = s;
    zero_out[e / g] = z;
  }
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

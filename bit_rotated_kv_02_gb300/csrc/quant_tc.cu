// Bulk rotate -> clip -> quantize -> pack on the tensor cores (tcgen05 MMA, TMA, tensor memory).
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": the long middle of a
// prompt is rotated by the per-head matrix R, clipped, quantized per group to 2 bits with a bf16 scale
// and zero point, and packed four codes per byte.  The result is the one the per-vector exact
// arithmetic gives (x_hat = float32 nearest to the exact x . R; lo = c*min, hi = c*max,
// scale = bf16((hi-lo)/3), zero = bf16(lo), code = clamp(rint((x_hat-zero)/scale), 0, 3)):
//
// 1. Tensor cores: a tile of 128 token rows of one KV head times R, with R split into two bf16
//    matrices R_hi = bf16(R), R_lo = bf16(R - R_hi) and x (bf16, exact) used against both: one
//    M=128, N=128, K=256 product accumulated in fp32 in tensor memory.
// 2. Bound: |x . R_j - acc_j| <= E = ||x||_2 * (kappa * || |R_hi,j| + |R_lo,j| ||_2 + ||Delta_j||_2),
//    Delta = R - R_hi - R_lo (exact in bf16), by Cauchy-Schwarz on the split residual plus the
//    tensor core's fp32 accumulation error, taken as kappa = 2^-17 times the sum of |products|.  The
//    accumulation order and truncation inside the tensor core are not specified bit for bit; the
//    kappa used is more than 5x the largest error measured on this hardware over 25 million dot
//    products of three value distributions (worst 2^-19.5).
// 3. Decisions from intervals: a group's scale and zero are taken from [acc - E, acc + E] when every
//    end point gives the same bf16 values, and a code when its distance from the rounding boundary
//    exceeds the bound carried through the quantizer's float32 steps.
// 4. Undecided elements are re-evaluated one by one by a warp: an fp32 compensated dot product
//    (error-free products and sums, Ogita-Rump-Oishi Dot2) over the exact R rebuilt from
//    R_hi + R_lo + Delta gives an interval of at most a few float32 ulps around x_hat; if that still
//    leaves the decision open, the float64 double-double / 128-bit integer evaluation decides.
//
// Warp roles (448 threads, one CTA per SM): warp 0 issues TMA loads of x tiles into a 4-stage ring,
// warp 1 owns tensor memory and issues the MMAs into 4 accumulators of 128 columns, warps 2-13 form
// three epilogue groups of four warps that take every third tile (the epilogue bounds the kernel: a
// third group adds latency hiding; two groups ran 7% slower); in an epilogue warp each thread owns one
// token row.  Each CTA processes a contiguous range of (head, tile) units; the R image in shared
// memory is rebuilt when the range crosses into the next head.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "oscar_internal.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int TILE = 128;                      // token rows per tile (MMA M)
constexpr int NSTAGE = 4;                      // x tiles in flight
constexpr int ATOM = 16384;                    // one 128-row x 64-channel bf16 swizzled atom
constexpr int STAGE_BYTES = 2 * ATOM;          // a tile: channels 0-63 and 64-127
constexpr int NACC = 4;                        // fp32 accumulators of 128 TMEM columns
constexpr int TMEM_COLS = NACC * 128;
constexpr int NGRP = 3;                        // epilogue groups of four warps
constexpr int THREADS = 64 + 128 * NGRP;
constexpr int EPI_THREADS = 128 * NGRP;
constexpr int DL_STRIDE = 130;                 // bf16 per row of the Delta table (spreads banks)
constexpr float KAPPA_TC = 0x1p-17f;
constexpr float MAGIC = 12582912.0f;           // 1.5 * 2^23: adding it rounds [0, 3] to an integer
constexpr uint32_t PACK_BIAS = 0x4B400000u * 0x55555555u;  // bits(MAGIC) * sum_k 4^k (mod 2^32)

constexpr int OFF_B = 0;                                   // [R_lo | R_hi] image: atoms 0,1 R_hi, 2,3 R_lo
constexpr int OFF_A = OFF_B + 4 * ATOM;                    // x ring
constexpr int OFF_DL = OFF_A + NSTAGE * STAGE_BYTES;       // Delta, bf16 [j][i]
constexpr int OFF_BAR = OFF_DL + D * DL_STRIDE * 2;
constexpr int OFF_PART = OFF_BAR + 256;                    // column sums of one half of the rows
constexpr int OFF_MISC = OFF_PART + 2 * D * 4;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;           // + slack to align the base to 1024
static_assert(OFF_BAR % 8 == 0 && (2 * NSTAGE + 2 * NACC + 1) * 8 <= 256, "barrier block");
static_assert(SMEM_BYTES <= 232448, "shared memory per block");

// misc words
constexpr int M_TMEM = 0, M_ABORT = 1, M_TABLE_EXACT = 3, M_RED = 4;

struct QArgs {
  int64_t n, T, U;  // rows, tiles per head, units (head, tile)
  int Hkv, num_pages;
  const float *R32, *clip;
  uint8_t *codes;
  uint16_t *scale, *zero;
  const int32_t *pt;
  uint32_t *err, *stats;
};

__device__ __forceinline__ float bfv(uint32_t b16) { return __uint_as_float(b16 << 16); }
__device__ __forceinline__ uint32_t lds_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

__device__ __forceinline__ bool aborted(const uint32_t *misc) {
  return *reinterpret_cast<const volatile uint32_t *>(misc + M_ABORT) != 0;
}
__device__ void report(const QArgs &a, uint32_t *misc, uint32_t bits) {
  *reinterpret_cast<volatile uint32_t *>(misc + M_ABORT) = 1;
  if (a.err) atomicOr(a.err, bits);
  if (a.stats) atomicOr(a.stats + 3, bits);
}
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, const QArgs &a, uint32_t *misc) {
  if (mbar_wait_bounded(bar, parity)) return true;
  report(a, misc, OSCAR_DEVERR_TIMEOUT);
  return false;
}

__device__ __forceinline__ void two_sum_f(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (s0, s1) += (lo^2, hi^2) of the two bf16 values packed in w (one paired float32 FMA).
__device__ __forceinline__ void sq2_acc(float &s0, float &s1, uint32_t w) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
  asm("{\n .reg .b64 x, c;\n mov.b64 x, {%2, %3};\n mov.b64 c, {%0, %1};\n fma.rn.f32x2 c, x, x, c;\n mov.b64 {%0, %1}, c;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "f"(lo), "f"(hi));
}
// 64 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),
        "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),
        "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
// Paired float32 operations (two lanes of a 64-bit register pair, one instruction).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 A, B, C, R;\n mov.b64 A, {%2, %3};\n mov.b64 B, {%4, %5};\n mov.b64 C, {%6, %7};\n"
      " fma.rn.f32x2 R, A, B, C;\n mov.b64 {%0, %1}, R;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 A, B, R;\n mov.b64 A, {%2, %3};\n mov.b64 B, {%4, %5};\n sub.rn.f32x2 R, A, B;\n mov.b64 {%0, %1}, R;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// min and max of 32 values by a three-input tree (depth 4).
__device__ __forceinline__ void minmax32(const float (&v)[32], float &mn, float &mx) {
  float a[11], b[11];
#pragma unroll
  for (int k = 0; k < 10; ++k) {
    a[k] = min3f(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
    b[k] = max3f(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  }
  a[10] = fminf(v[30], v[31]);
  b[10] = fmaxf(v[30], v[31]);
  mn = fminf(min3f(min3f(a[0], a[1], a[2]), min3f(a[3], a[4], a[5]), min3f(a[6], a[7], a[8])), fminf(a[9], a[10]));
  mx = fmaxf(max3f(max3f(b[0], b[1], b[2]), max3f(b[3], b[4], b[5]), max3f(b[6], b[7], b[8])), fmaxf(b[9], b[10]));
}

// x_i of tile row `row` (bf16 in the swizzled stage).
__device__ __forceinline__ float stage_x(const uint8_t *st, int row, int i) {
  return bfv(lds_u16(st + (i >> 6) * ATOM + sw128_offset(row, i & 63)));
}

// Warp-cooperative interval for x_hat of (row, column j): [x, y] contains the float32 nearest to the
// exact x . R_j.  Products are split error-free (p + e = x r, FMA), partial sums carry their rounding
// errors (TwoSum), and the errors are summed in plain float32, whose own error is below
// gamma_2n * gamma_n * sum|x r| < 2^-33 sum|x r|; the interval uses 2^-31 times the computed sum.
// Every lane ends with the same values (the butterfly's operations are symmetric in the partners).
// Out of line and single-item: it runs for a few elements per tile and must not crowd the
// instruction cache.
__device__ __noinline__ float2 dot2_interval(const uint8_t *st, const uint8_t *sm, const float *Rg, bool table_exact,
                                            int row, int j) {
  const int lane = threadIdx.x & 31;
  const uint16_t *Dl = reinterpret_cast<const uint16_t *>(sm + OFF_DL);
  float s = 0.f, c = 0.f, sab = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k, at = k >> 1, kk = i & 63;
    const float xv = bfv(lds_u16(st + at * ATOM + sw128_offset(row, kk)));
    float rv;
    if (table_exact) {
      const int off = sw128_offset(j, kk);
      rv = __fadd_rn(__fadd_rn(bfv(lds_u16(sm + OFF_B + at * ATOM + off)), bfv(lds_u16(sm + OFF_B + (2 + at) * ATOM + off))),
                     bfv(Dl[j * DL_STRIDE + i]));
    } else {
      rv = Rg[i * D + j];
    }
    const float p = __fmul_rn(xv, rv);
    const float e = fmaf(xv, rv, -p);
    float tt, qq;
    two_sum_f(s, p, tt, qq);
    s = tt;
    c = __fadd_rn(c, __fadd_rn(qq, e));
    sab = fmaf(fabsf(xv), fabsf(rv), sab);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float s2 = __shfl_xor_sync(FULL, s, off);
    const float c2 = __shfl_xor_sync(FULL, c, off);
    const float a2 = __shfl_xor_sync(FULL, sab, off);
    float tt, qq;
    two_sum_f(s, s2, tt, qq);
    s = tt;
    c = __fadd_rn(__fadd_rn(c, c2), qq);
    sab = __fadd_rn(sab, a2);
  }
  float hi, lo;
  two_sum_f(s, c, hi, lo);
  const float B = __fadd_ru(__fmul_ru(sab, 0x1p-31f), 1e-36f);
  return make_float2(__fadd_rd(hi, __fsub_rd(lo, B)), __fadd_ru(hi, __fadd_ru(lo, B)));
}

// Next pending item (lane, bit) of the per-lane masks, lowest lane first, removed from the mask;
// every lane returns the same pair.  Call only while some lane's mask is non-zero.
__device__ __forceinline__ int2 next_item(uint32_t &pend) {
  const int sl = __ffs(__ballot_sync(FULL, pend != 0)) - 1;
  const int k = __ffs(__shfl_sync(FULL, pend, sl)) - 1;
  if ((int)(threadIdx.x & 31) == sl) pend &= pend - 1;
  return make_int2(sl, k);
}

// ||x||_2 bound factor of a tile row: E = cE * ||x||_2, rounded up (the row read from the stage).
__device__ __forceinline__ float row_bound(const uint8_t *st, int row, float cE) {
  float sq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int at = 0; at < 2; ++at) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 w = *reinterpret_cast<const uint4 *>(st + at * ATOM + (row >> 3) * 1024 + (row & 7) * 128 +
                                                       ((q ^ (row & 7)) << 4));
      sq2_acc(sq[0], sq[1], w.x);
      sq2_acc(sq[2], sq[3], w.y);
      sq2_acc(sq[4], sq[5], w.z);
      sq2_acc(sq[6], sq[7], w.w);
    }
  }
  const float ss = ((sq[0] + sq[1]) + (sq[2] + sq[3])) + ((sq[4] + sq[5]) + (sq[6] + sq[7]));
  // 1 + 2^-14 covers the float32 sum of squares; 1e-36 covers squares that underflow.
  return __fadd_ru(__fmul_ru(cE, __fsqrt_ru(__fadd_ru(__fmul_ru(ss, 1.0f + 0x1p-14f), 1e-36f))), 1e-37f);
}

// Rebuild the shared-memory image of head h's R (epilogue threads tb in [0, 256) build it, the rest of
// the epilogue threads only take part in the barriers): the MMA operand
// [R_hi ; R_lo]^T in swizzled K-major atoms, the residual table Delta, and the bound constant cE.
__device__ void build_head(const QArgs &a, uint8_t *sm, uint32_t *misc, uint64_t *bready, int h, int tb) {
  named_bar_sync(1, EPI_THREADS);  // every tile of the previous head is finished (its MMAs complete)
  const int j = tb & (D - 1), half = tb >> 7;  // threads tb >= 256 only take part in the barriers
  bool exact = true;
  float sd = 0.f, sr = 0.f;
  float *part = reinterpret_cast<float *>(sm + OFF_PART);
  if (tb < 256) {
  const float *R = a.R32 + (size_t)h * D * D;
  uint8_t *Bs = sm + OFF_B;
  uint16_t *Dl = reinterpret_cast<uint16_t *>(sm + OFF_DL);
  float rr[D / 2];
#pragma unroll
  for (int m = 0; m < D / 2; ++m) rr[m] = R[(2 * m + half) * D + j];  // all loads in flight at once
#pragma unroll
  for (int m = 0; m < D / 2; ++m) {
    const int i = 2 * m + half;
    const float r = rr[m];
    const uint16_t rh = f32_to_bf16(r);
    const float rem = __fsub_rn(r, bfv(rh));
    const uint16_t rl = f32_to_bf16(rem);
    const float dl = __fsub_rn(rem, bfv(rl));
    const uint16_t db = f32_to_bf16(dl);
    exact = exact && bfv(db) == dl && __fadd_rn(__fadd_rn(bfv(rh), bfv(rl)), bfv(db)) == r;
    const int at = i >> 6, off = sw128_offset(j, i & 63);
    *reinterpret_cast<uint16_t *>(Bs + at * ATOM + off) = rh;
    *reinterpret_cast<uint16_t *>(Bs + (2 + at) * ATOM + off) = rl;
    Dl[j * DL_STRIDE + i] = db;
    sd = fmaf(dl, dl, sd);
    const float t = __fadd_rn(fabsf(bfv(rh)), fabsf(bfv(rl)));
    sr = fmaf(t, t, sr);
  }
  if (half) {
    part[j] = sd;
    part[D + j] = sr;
  }
  }
  fence_proxy_async_smem();
  const bool all_exact = named_bar_and(1, EPI_THREADS, exact);
  if (tb == 0) {
    misc[M_TABLE_EXACT] = all_exact ? 1u : 0u;
    mbar_arrive(bready);
  }
  if (tb < 128) {
    // per-column bound factor, every step rounded up; 1 + 2^-12 covers the float32 sums above
    const float ssr = __fmul_ru(__fadd_ru(sr, part[D + j]), 1.0f + 0x1p-12f);
    const float ssd = __fmul_ru(__fadd_ru(sd, part[j]), 1.0f + 0x1p-12f);
    float v = __fadd_ru(__fmul_ru(KAPPA_TC, __fsqrt_ru(ssr)), __fsqrt_ru(ssd));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, off));
    if ((tb & 31) == 0) reinterpret_cast<float *>(misc)[M_RED + (tb >> 5)] = v;
  }
  named_bar_sync(1, EPI_THREADS);
}

// The exact x_hat of (row, j) by the float64 double-double / 128-bit integer evaluation (warp-wide).
__device__ __noinline__ float exact_value(const uint8_t *st, const float *Rg, int row, int j, bool &unproven) {
  return exact_rot_elem_f([st, row](int i) { return stage_x(st, row, i); }, Rg, j, unproven);
}

// a[gi] for a small per-group register array, without dynamic register indexing.
template <int NG, class T>
__device__ __forceinline__ T pick(const T (&a)[NG], int gi) {
  T r = a[0];
#pragma unroll
  for (int k = 1; k < NG; ++k)
    if (gi == k) r = a[k];
  return r;
}

// One tile in an epilogue thread, which owns row quad*32 + lane of the tile (E: its fast-path bound).
// Per-group values are picked from registers in rolled chunk loops and the rare float64 evaluation is
// out of line, so that the code of both epilogue groups fits the instruction cache.
template <int G>
__device__ void epilogue_tile(const QArgs &a, const uint8_t *sm, const uint8_t *st, uint32_t tbase, int h, int64_t t,
                              int quad, float E, bool table_exact, float clip, QuantStats &stt) {
  constexpr int NG = D / G, CPG = G / 32;  // groups per row, 32-column chunks per group
  const int lane = threadIdx.x & 31, row = quad * 32 + lane;
  const float *Rg = a.R32 + (size_t)h * D * D;

  // ---- output row ----
  const int64_t r = t * TILE + row;
  bool store = r < a.n;
  size_t orow = 0;
  if (store) {
    if (a.pt == nullptr) {
      orow = (size_t)r * a.Hkv + h;
    } else {
      const int page = a.pt[r / PAGE];
      store = page >= 0 && page < a.num_pages;
      if (!store && a.err) atomicOr(a.err, OSCAR_DEVERR_PAGE_INDEX);
      orow = store ? ((size_t)page * a.Hkv + h) * PAGE + (size_t)(r % PAGE) : 0;
    }
  }

  // ---- pass 1: chunk and group extremes of the tensor-core values ----
  float cmn[4], cmx[4], mn[NG], mx[NG];
#pragma unroll
  for (int hlf = 0; hlf < 2; ++hlf) {
    float v[64];
    tmem_ld64(tbase + 64 * hlf, v);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      float w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = v[32 * cc + i];
      minmax32(w, cmn[2 * hlf + cc], cmx[2 * hlf + cc]);
    }
  }
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    mn[gi] = cmn[gi * CPG];
    mx[gi] = cmx[gi * CPG];
#pragma unroll
    for (int k = 1; k < CPG; ++k) {
      mn[gi] = fminf(mn[gi], cmn[gi * CPG + k]);
      mx[gi] = fmaxf(mx[gi], cmx[gi * CPG + k]);
    }
  }
  // Every end point of [mn - E, mn + E] and [mx - E, mx + E] must give the same bf16 zero / scale
  // (zero is increasing in the minimum; scale increasing in the maximum, decreasing in the minimum).
  float mnlo[NG], mnhi[NG], mxlo[NG], mxhi[NG];
  uint16_t zq[NG], sq16[NG];
  bool uz[NG], us[NG], any_und = false;
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    mnlo[gi] = __fsub_rd(mn[gi], E);
    mnhi[gi] = __fadd_ru(mn[gi], E);
    mxlo[gi] = __fsub_rd(mx[gi], E);
    mxhi[gi] = __fadd_ru(mx[gi], E);
    zq[gi] = zero_of(clip, mnlo[gi]);
    uz[gi] = zq[gi] != zero_of(clip, mnhi[gi]);
    sq16[gi] = scale_of(clip, mnhi[gi], mxlo[gi]);
    us[gi] = sq16[gi] != scale_of(clip, mnlo[gi], mxhi[gi]);
    any_und |= uz[gi] || us[gi];
    stt.exact_groups += __popc(__ballot_sync(FULL, uz[gi] || us[gi]));
  }

  // ---- exact extremes of undecided groups: Dot2 intervals, then float64 / integer if still open ----
  // Only elements whose interval reaches the group's extreme can be the extreme: v <= mn + 2E for the
  // minimum (needed by zero and scale), v >= mx - 2E for the maximum (needed by scale).
  if (__any_sync(FULL, any_und)) {
    float tmin[NG], tmax[NG], emnlo[NG], emnhi[NG], emxlo[NG], emxhi[NG];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      tmin[gi] = (uz[gi] || us[gi]) ? __fadd_ru(mnhi[gi], E) : -INFINITY;
      tmax[gi] = us[gi] ? __fsub_rd(mxlo[gi], E) : INFINITY;
      emnlo[gi] = emnhi[gi] = INFINITY;
      emxlo[gi] = emxhi[gi] = -INFINITY;
    }
#pragma unroll 1
    for (int tier = 0; tier < 2; ++tier) {
      bool unproven = false;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int gi = c / CPG;
        const float lim_min = pick(tmin, gi), lim_max = pick(tmax, gi);
        const bool may = pick(cmn, c) <= lim_min || pick(cmx, c) >= lim_max;
        if (!__any_sync(FULL, may)) continue;
        float v[32];
        tmem_ld32(tbase + 32 * c, v);
        uint32_t cm = 0, cx = 0;
        if (may) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (v[i] <= lim_min) cm |= 1u << i;
            if (v[i] >= lim_max) cx |= 1u << i;
          }
        }
        float lmnlo = INFINITY, lmnhi = INFINITY, lmxlo = -INFINITY, lmxhi = -INFINITY;
        uint32_t pend = cm | cx;
        while (__any_sync(FULL, pend != 0)) {
          const int2 it2 = next_item(pend);
          const int srow = quad * 32 + it2.x, j = 32 * c + it2.y;
          float2 iv;
          if (tier == 0) iv = dot2_interval(st, sm, Rg, table_exact, srow, j);
          else iv.x = iv.y = exact_value(st, Rg, srow, j, unproven);
          if (lane == it2.x) {
            if ((cm >> it2.y) & 1u) { lmnlo = fminf(lmnlo, iv.x); lmnhi = fminf(lmnhi, iv.y); }
            if ((cx >> it2.y) & 1u) { lmxlo = fmaxf(lmxlo, iv.x); lmxhi = fmaxf(lmxhi, iv.y); }
          }
          ++stt.exact_elems;
        }
#pragma unroll
        for (int gi2 = 0; gi2 < NG; ++gi2) {
          if (gi2 == gi) {
            emnlo[gi2] = fminf(emnlo[gi2], lmnlo);
            emnhi[gi2] = fminf(emnhi[gi2], lmnhi);
            emxlo[gi2] = fmaxf(emxlo[gi2], lmxlo);
            emxhi[gi2] = fmaxf(emxhi[gi2], lmxhi);
          }
        }
      }
      if (__any_sync(FULL, unproven)) ++stt.unproven;
      bool still = false;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        if (uz[gi]) {
          const uint16_t z = zero_of(clip, emnlo[gi]);
          if (z == zero_of(clip, emnhi[gi]) || tier == 1) { zq[gi] = z; uz[gi] = false; }
        }
        if (us[gi]) {
          const uint16_t s = scale_of(clip, emnhi[gi], emxlo[gi]);
          if (s == scale_of(clip, emnlo[gi], emxhi[gi]) || tier == 1) { sq16[gi] = s; us[gi] = false; }
        }
        if (uz[gi] || us[gi]) {
          emnlo[gi] = emnhi[gi] = INFINITY;
          emxlo[gi] = emxhi[gi] = -INFINITY;
          still = true;
        }
      }
      if (!__any_sync(FULL, still)) break;
    }
  }

  // ---- pass 2: codes ----
  // u3 = sat(acc * (1/s)/3 - (z/s)/3) and 3*u3 is within delta of clamp((x_hat - z)/s, 0, 3) as the
  // quantizer computes it in float32; a code is taken from 3*u3 when it lies more than delta inside
  // (k - 1/2, k + 1/2), else the element is re-evaluated.
  float zf[NG], sf[NG], inv3[NG], c03[NG], thr[NG];
  bool valid[NG];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    zf[gi] = bfv(zq[gi]);
    sf[gi] = bfv(sq16[gi]);
    valid[gi] = sf[gi] != 0.0f && isfinite(sf[gi]);
    const float inv = valid[gi] ? __frcp_rn(sf[gi]) : 0.0f;
    inv3[gi] = __fdiv_rn(inv, 3.0f);
    c03[gi] = __fdiv_rn(-__fmul_rn(zf[gi], inv), 3.0f);
    const float Mg = fmaxf(fabsf(mnlo[gi]), fabsf(mxhi[gi]));
    const float delta = __fadd_ru(__fmul_ru(__fadd_ru(E, __fmul_ru(0x1p-19f, __fadd_ru(Mg, fabsf(zf[gi])))),
                                            __fmul_ru(inv, 1.0f + 0x1p-19f)),
                                  0x1p-17f);
    thr[gi] = __fsub_rd(0.5f, delta);
  }
  uint2 *cdst = reinterpret_cast<uint2 *>(a.codes + orow * (D / 4));
  const float2 three = make_float2(3.0f, 3.0f), magic = make_float2(MAGIC, MAGIC);
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    const int gi = c / CPG;
    const float ginv3 = pick(inv3, gi), gc03 = pick(c03, gi), gthr = pick(thr, gi);
    float v[32];
    tmem_ld32(tbase + 32 * c, v);
    uint32_t bm[32];
    float dd[32];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 u3 = make_float2(fma_sat(v[i], ginv3, gc03), fma_sat(v[i + 1], ginv3, gc03));
      const float2 m = fma2(u3, three, magic);        // MAGIC + rint(3 u3)
      const float2 d = fma2(u3, three, sub2(magic, m));  // 3 u3 - rint(3 u3)
      dd[i] = d.x;
      dd[i + 1] = d.y;
      bm[i] = __float_as_uint(m.x);
      bm[i + 1] = __float_as_uint(m.y);
    }
    // pack 16 codes per word: sum of bits(m_i) << 2i by a tree (bits(m_i) = bits(MAGIC) + code_i)
    uint32_t p[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) p[k] = bm[2 * k] + (bm[2 * k + 1] << 2);
#pragma unroll
    for (int k = 0; k < 8; ++k) p[k] = p[2 * k] + (p[2 * k + 1] << 4);
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = p[2 * k] + (p[2 * k + 1] << 8);
    uint32_t w0 = p[0] + (p[1] << 16) - PACK_BIAS, w1 = p[2] + (p[3] << 16) - PACK_BIAS;
    float e[11];
#pragma unroll
    for (int k = 0; k < 10; ++k) e[k] = max3abs(dd[3 * k], dd[3 * k + 1], dd[3 * k + 2]);
    e[10] = max3abs(dd[30], dd[31], 0.0f);
    const float dmax = max3f(max3f(e[0], e[1], e[2]), max3f(e[3], e[4], e[5]), max3f(max3f(e[6], e[7], e[8]), e[9], e[10]));
    if (__any_sync(FULL, !(dmax < gthr))) {
      uint32_t near = 0;
      if (!(dmax < gthr)) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (!(fabsf(dd[i]) < gthr)) near |= 1u << i;
      }
      const float gz = pick(zf, gi), gs = pick(sf, gi);
      const bool gvalid = pick(valid, gi);
      while (__any_sync(FULL, near != 0)) {
        const int2 it2 = next_item(near);
        const int srow = quad * 32 + it2.x, j = 32 * c + it2.y;
        const float2 iv = dot2_interval(st, sm, Rg, table_exact, srow, j);
        // the owning lane's scale/zero decide; its verdict is broadcast so the warp stays converged
        int code = code_of(iv.x, gz, gs, gvalid);
        if (__shfl_sync(FULL, code != code_of(iv.y, gz, gs, gvalid), it2.x)) {
          bool unproven = false;
          code = code_of(exact_value(st, Rg, srow, j, unproven), gz, gs, gvalid);
          if (__any_sync(FULL, unproven)) ++stt.unproven;
        }
        if (lane == it2.x) {
          const int k = it2.y;
          if (k < 16) w0 = (w0 & ~(3u << (2 * k))) | ((uint32_t)code << (2 * k));
          else w1 = (w1 & ~(3u << (2 * (k - 16)))) | ((uint32_t)code << (2 * (k - 16)));
        }
        ++stt.exact_elems;
      }
    }
    if (store) cdst[c] = make_uint2(w0, w1);
  }

  // ---- scale and zero ----
  if (store) {
    if constexpr (NG == 1) {
      a.scale[orow] = sq16[0];
      a.zero[orow] = zq[0];
    } else if constexpr (NG == 2) {
      reinterpret_cast<uint32_t *>(a.scale)[orow] = sq16[0] | ((uint32_t)sq16[1] << 16);
      reinterpret_cast<uint32_t *>(a.zero)[orow] = zq[0] | ((uint32_t)zq[1] << 16);
    } else {
      reinterpret_cast<uint2 *>(a.scale)[orow] =
          make_uint2(sq16[0] | ((uint32_t)sq16[1] << 16), sq16[2] | ((uint32_t)sq16[3] << 16));
      reinterpret_cast<uint2 *>(a.zero)[orow] =
          make_uint2(zq[0] | ((uint32_t)zq[1] << 16), zq[2] | ((uint32_t)zq[3] << 16));
    }
  }
}

template <int G>
__global__ void __launch_bounds__(THREADS, 1) quant_tc_kernel(const __grid_constant__ CUtensorMap xmap, QArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
  uint64_t *full = bars, *empty = bars + NSTAGE, *accf = bars + 2 * NSTAGE, *acce = bars + 2 * NSTAGE + NACC;
  uint64_t *bready = bars + 2 * NSTAGE + 2 * NACC;
  uint32_t *misc = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 4); }
    for (int b = 0; b < NACC; ++b) { mbar_init(accf + b, 1); mbar_init(acce + b, 4); }
    mbar_init(bready, 1);
    misc[M_ABORT] = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(misc + M_TMEM, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[M_TMEM];
  const int64_t u0 = a.U * blockIdx.x / gridDim.x, u1 = a.U * (blockIdx.x + 1) / gridDim.x;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      for (int64_t u = u0; u < u1; ++u, ++it) {
        const uint32_t s = it % NSTAGE;
        if (aborted(misc) || !wait_or_abort(empty + s, ((it / NSTAGE) & 1u) ^ 1u, a, misc)) break;
        mbar_arrive_expect_tx(full + s, STAGE_BYTES);
        const int h = (int)(u / a.T), t0 = (int)(u % a.T) * TILE;
        uint8_t *dst = sm + OFF_A + s * STAGE_BYTES;
        tma_load_3d(dst, &xmap, 0, h, t0, full + s);
        tma_load_3d(dst + ATOM, &xmap, 64, h, t0, full + s);
      }
      if (aborted(misc))  // copies still in flight must land before the block exits
        for (uint32_t k = it > NSTAGE ? it - NSTAGE : 0; k < it; ++k)
          mbar_wait_bounded(full + k % NSTAGE, (k / NSTAGE) & 1u, 100000000ull);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t IDESC = umma_idesc_bf16(TILE, D);
      uint32_t it = 0, seg = 0;
      bool ok = true;
      for (int64_t u = u0; u < u1 && ok; ++seg) {
        const int64_t seg_end = min(u1, (u / a.T + 1) * a.T);
        if (!wait_or_abort(bready, seg & 1u, a, misc)) break;
        for (; u < seg_end; ++u, ++it) {
          const uint32_t s = it % NSTAGE, b = it % NACC;
          if (aborted(misc) || !wait_or_abort(full + s, (it / NSTAGE) & 1u, a, misc) ||
              !wait_or_abort(acce + b, ((it / NACC) & 1u) ^ 1u, a, misc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t *A = sm + OFF_A + s * STAGE_BYTES;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            // lo half first (smaller terms first), then hi; each half: 2 atoms x 4 K-steps of 16
            const int kq = q & 7, at = kq >> 2, off = (kq & 3) * 32;
            const int batom = (q < 8) ? 2 + at : at;
            umma_bf16(tmem + b * 128, umma_desc_sw128(A + at * ATOM + off), umma_desc_sw128(sm + OFF_B + batom * ATOM + off),
                      IDESC, q > 0 ? 1u : 0u);
          }
          umma_commit(accf + b);
        }
      }
      if (it > 0)  // the last commit covers every MMA issued: let them finish before tensor memory is freed
        mbar_wait_bounded(accf + (it - 1) % NACC, ((it - 1) / NACC) & 1u);
    }
  } else {
    // ---------------- epilogue groups ----------------
    const int ew = warp - 2, grp = ew >> 2, quad = warp & 3, tb = tid - 64;
    QuantStats stt{0, 0, 0};
    uint32_t it = 0;
    for (int64_t u = u0; u < u1;) {
      const int h = (int)(u / a.T);
      const int64_t seg_end = min(u1, (int64_t)(h + 1) * a.T);
      build_head(a, sm, misc, bready, h, tb);
      const float *red = reinterpret_cast<const float *>(misc) + M_RED;
      const float cE = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
      const bool table_exact = misc[M_TABLE_EXACT] != 0;
      const float clip = a.clip[h];
      for (; u < seg_end; ++u, ++it) {
        // decisions stay warp-uniform: the tensor-memory loads below are warp-collective
        if ((int)(it % NGRP) != grp || __any_sync(FULL, aborted(misc))) continue;
        const uint32_t s = it % NSTAGE, b = it % NACC;
        // the row norm needs only the loaded tile: compute it while the MMA runs
        if (!__all_sync(FULL, wait_or_abort(full + s, (it / NSTAGE) & 1u, a, misc))) continue;
        const uint8_t *st = sm + OFF_A + s * STAGE_BYTES;
        const float E = row_bound(st, quad * 32 + lane, cE);
        if (!__all_sync(FULL, wait_or_abort(accf + b, (it / NACC) & 1u, a, misc))) continue;
        tc_fence_after();
        epilogue_tile<G>(a, sm, st, tmem + ((uint32_t)(quad * 32) << 16) + b * 128, h, u % a.T, quad, E,
                         table_exact, clip, stt);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(acce + b);
          mbar_arrive(empty + s);
        }
      }
    }
    flush_stats(a.stats, stt);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

namespace {

template <int G>
cudaError_t launch_g(const CUtensorMap &map, const QArgs &a, int grid, cudaStream_t s) {
  const cudaError_t e = cudaFuncSetAttribute(quant_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  quant_tc_kernel<G><<<grid, THREADS, SMEM_BYTES, s>>>(map, a);
  return cudaGetLastError();
}

}  // namespace

// Rows [0, n) of x (bf16, row r of head h at x + r * x_row_stride + h * 128) -> codes, scale, zero of
// rows r * Hkv + h (pt == nullptr) or of page pt[r / 64], slot r % 64 (pt != nullptr).
cudaError_t launch_quantize_rows(int64_t n, int Hkv, int g, const uint16_t *x, int64_t x_row_stride, const float *R32,
                                 const float *clip, uint8_t *codes, uint16_t *scale, uint16_t *zero,
                                 const int32_t *pt, int num_pages, uint32_t *err, uint32_t *stats, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n > (int64_t)INT32_MAX - TILE || Hkv <= 0) {
    set_last_error("quantize: row count out of range");
    return cudaErrorInvalidValue;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) {
    set_last_error("quantize: cuTensorMapEncodeTiled unavailable from the driver");
    return cudaErrorNotSupported;
  }
  CUtensorMap map;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)n};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)x_row_stride * 2};
  cuuint32_t box[3] = {64, 1, TILE}, estr[3] = {1, 1, 1};
  const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(x), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("quantize: tensor map rejected (x must be 16-byte aligned with a row stride multiple of 8)");
    return cudaErrorInvalidValue;
  }
  QArgs a;
  a.n = n;
  a.T = (n + TILE - 1) / TILE;
  a.U = a.T * Hkv;
  a.Hkv = Hkv;
  a.num_pages = num_pages;
  a.R32 = R32;
  a.clip = clip;
  a.codes = codes;
  a.scale = scale;
  a.zero = zero;
  a.pt = pt;
  a.err = err;
  a.stats = stats;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = (int)(a.U < sms ? a.U : sms);
  switch (g) {
    case 32: return launch_g<32>(map, a, grid, s);
    case 64: return launch_g<64>(map, a, grid, s);
    case 128: return launch_g<128>(map, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oscar

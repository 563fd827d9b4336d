// Decode attention over the three-segment pool on the 5th-generation tensor cores (tcgen05, TMEM, bulk
// async copies), uniform INT2 levels, group sizes 32, 64 and 128.
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": the INT2 kernel unpacks
// the 2-bit codes, dequantizes with scale and zero point and accumulates in floating point; a BF16 kernel
// handles the sink and the recent window; an online-softmax merge combines the parts.
// "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract: a custom
// INT2 attention kernel compatible with paged KV-cache serving.
//
// Launches (all with programmatic dependent launch on the caller's stream):
//   qrot_kernel  per (sequence, KV head): q_rot = q . R_k for the G query heads and the image of the Q.K
//                B operand (six base-16 digit planes of the fixed-point q_rot in e4m3, or its fp16 hi / lo
//                split; one set of columns per head and group) with the score factors, in the workspace.
//   hist_kernel  one CTA per SM over an equal share of the flattened (sequence, KV head, page) space, in
//                tiles of 128 tokens (two pages of one segment):
//                  warp 0      bulk-copies pages (codes, scale/zero rows) into a ring and, per segment, the
//                              Q.K operand image;
//                  warp 1      allocates tensor memory and issues the MMAs (one thread): Q.K up to two tiles
//                              ahead of P.V, one commit per Q.K and one per P.V;
//                  warps 2-5   unpack each token's 128 K codes (e4m3 or fp16) into tensor memory, the A
//                              operand of Q.K (M = 128 tokens, K = 128 channels), and copy its scale/zero
//                              rows into a small ring for the softmax;
//                  warps 6-9   unpack the V codes into a 128-byte-swizzled shared-memory tile, read as the
//                              MN-major A operand of P.V (M = 128 channels, K = 128 tokens);
//                  warps 10-17 two softmax warpgroups, each over half of the G query heads of every tile
//                              (one token row per thread): scores from tensor memory, online softmax, the
//                              weights (fp16 hi + lo) as the B operand of P.V, and each segment's flush into
//                              a partial (m, l, o_rot).
//   bf16_kernel  the BF16 sink/window partials and, in the decode step, the demotion (part::bf16_role).
//   merge        v1::merge_kernel: LSE merge, o . R_v^T, normalisation (decode step: append, counters).
//
// Exactness of the tensor-core sums.  q_rot * 2^sigma is taken on a fixed-point grid with 24 significant
// bits (y = q_rot 2^sigma, |y| < 2^14).  fp16 form: a 2-bit code c in the low mantissa bits of an fp16 with a
// zero exponent field is the subnormal c * 4^k * 2^-24 (k = its 2-bit position in the 16-bit lane), so one
// AND places two codes; hi = 8 rint(y / 8), lo = rint((y - hi) 256) / 256, each scaled by 4^-k, so every
// product with a code is an integer multiple of 2^-21 (hi) or 2^-32 (lo) and a token's 128 products stay below
// 2^24 such units.  e4m3 form (kind::f8f6f4, K = 32 per MMA): a code in the two low bits of a byte is c * 2^-9,
// two bits up c * 2^-7; the integer Y = y 2^9 is written as six balanced base-16 digits d_t (|d_t| <= 8, exact
// in e4m3), one column per digit plane, so each plane's sum is a small integer multiple of 2^-9 and the score
// is 2^(-sigma - 2) sum_t 16^t S_t (Horner in float32).  Either way the float32 accumulation of Q.K is exact
// in any order, and
//   score = kf * sum_g scale_g * S_g + sum_g zero_g * zf_g,
//   o_rot[ch] = 2^(24 - 2k - tau) * (O_hi + O_lo)[ch] + sum_t p_t zero_t,g(ch),
// with weights p * scale * 2^tau split into fp16 hi + lo (22 significant bits) and a lazily rescaled base-2
// online softmax (the reference grows only when a score exceeds it by more than 2^LAZY).
#include <cuda_fp8.h>

#include "oscar_internal.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "bf16_part.cuh"
#include "split.cuh"

namespace oscar {

namespace tc {

constexpr int TILE = 128;
constexpr int W_PROD = 0, W_MMA = 1, W_V0 = 6, W_S0 = 10;  // K unpack warps: 2..5
constexpr int TI = 16;        // tile-information ring
constexpr int MR = 4;         // scale/zero ring: tiles in flight between the K unpack and the softmax
constexpr int LAZY = 16;      // the softmax reference grows only when a score exceeds it by more than 2^16
constexpr int WEXP = 14 - LAZY;
constexpr int TAU_HEAD = 2;   // the weight scale leaves the V scales 4x headroom before it must shrink
constexpr int OFF_KC = 0, OFF_VC = 2048, OFF_META = 4096;
constexpr int AV_BYTES = 2 * 16384;  // one 128 x 128 fp16 tile: two 64-channel atom columns

template <int G, int NG>
struct Cfg {
  // softmax warpgroups: each takes G / SG query heads of every tile (their columns of S and O, their rows of
  // the weight operand), so that the per-tile softmax work, the critical path of a tile, is split
  static constexpr int SG = G >= 2 ? 2 : 1;
  static constexpr int GH = G / SG;                                     // heads per softmax warpgroup
  static constexpr int THREADS = 64 + 256 + 128 * SG;
  // registers per thread: a CTA's warps are spread over the SM's four sub-partitions of 16K registers each,
  // so 18 warps (five on some sub-partitions) allow 96 per thread and 14 warps (four at most) 128
  static constexpr int MAXREG = SG == 2 ? 96 : 128;
  static constexpr int NCOL = 2 * G * NG;                               // used MMA columns
  static constexpr int N = NCOL <= 16 ? 16 : ((NCOL + 15) / 16) * 16;   // MMA N (M = 128 needs N % 16 == 0)
  static constexpr int NCG = N / SG;                                    // columns per softmax warpgroup
  static constexpr int META = 2 * NG;                                   // bytes per token of one of Ks/Kz/Vs/Vz
  static constexpr int PAGE_BYTES = 4096 + 4 * 64 * META;               // Kc | Vc | Ks | Kz | Vs | Vz
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
  // one Q.K operand buffer for N = 64 (eight heads x four groups), two otherwise, and a shorter ring there
  static constexpr int BQN = N >= 64 ? 1 : 2;
  static constexpr int RING = NG == 1 ? 7 : (N >= 64 ? 4 : 5);
  // Q.K in fp8 (kind::f8f6f4, e4m3, K = 32 per MMA) when the six digit planes of every head and group fit in
  // N <= 128 (an MMA of N <= 128 costs the same): K codes as e4m3 subnormals, q_rot as six base-16 digits.
  // Otherwise (eight heads x four groups) Q.K in fp16 with the hi / lo split (two columns per head and group).
  static constexpr int QT = 6;                                          // digit planes of q_rot
  static constexpr int NQG8 = ((GH * NG * QT + 7) / 8) * 8;
  static constexpr bool QK8 = SG * NQG8 <= 128;
  static constexpr int NQG = QK8 ? NQG8 : NCG;                          // S columns per softmax warpgroup
  static constexpr int NQ = QK8 ? ((SG * NQG8 + 15) / 16) * 16 : N;     // MMA N of Q.K
  static constexpr int AKC = QK8 ? 32 : 64;                             // TMEM columns of one K operand
  // fp16 Q.K with several groups: one MMA of N = 2G per 16-channel step into the columns of that step's group
  // (S column g 2G + 2h + term), so that no step multiplies the zero rows of the other groups' columns
  static constexpr bool QKG = !QK8 && NG > 1;
  static constexpr int BQ_FACTORS = ((G + G * NG) * 4 + 15) / 16 * 16;  // kf[G], zf[G][NG]
  static constexpr int BQ_IMG = QK8 ? NQ * 128 : N * 256;               // [NQ][128] e4m3 / [N][128] fp16
  static constexpr int BQ_BYTES = BQ_IMG + BQ_FACTORS;
  static constexpr int BW_BYTES = N * 256;
  // N = 64: the weight operand MN-major (token k's 64 columns form one 128-byte swizzled row, so that a thread
  // stores its columns with 16-byte stores); smaller N: K-major (column n's 128 tokens in two 128-byte rows)
  static constexpr bool BW_MN = N == 64;
  // tensor memory columns: K operands and S for NSQ tiles (Q.K runs two tiles ahead of P.V), O for two segments
  static constexpr int NSQ = 4 * (AKC + NQ) + 2 * N <= 512 ? 4 : 3;
  static constexpr int TM_AK = 0, TM_S = AKC * NSQ, TM_O = TM_S + NSQ * NQ;
  static constexpr int TM_USED = TM_O + 2 * N;
  static constexpr int TM_COLS = TM_USED <= 256 ? 256 : 512;
  // shared memory (the operand images at 1024-byte boundaries); V tiles: four where they fit, else three
  static constexpr int BQ_STRIDE0 = ((BQ_BYTES + 1023) / 1024) * 1024;
  static constexpr int REST = BQN * BQ_STRIDE0 + 2 * BW_BYTES + RING * STAGE_BYTES + MR * TILE * 4 * META + 4096;
  static constexpr int NAV = 4 * AV_BYTES + REST <= 227 * 1024 ? 4 : 3;
  static constexpr int OFF_AV = 0;
  static constexpr int OFF_BQ = OFF_AV + NAV * AV_BYTES;
  static constexpr int BQ_STRIDE = ((BQ_BYTES + 1023) / 1024) * 1024;
  static constexpr int OFF_BW = OFF_BQ + BQN * BQ_STRIDE;
  static constexpr int OFF_RING = OFF_BW + 2 * BW_BYTES;
  static constexpr int OFF_MRING = OFF_RING + RING * STAGE_BYTES;
  static constexpr int MRING_TILE = TILE * 4 * META;
  static constexpr int OFF_TINFO = OFF_MRING + MR * MRING_TILE;
  static constexpr int OFF_BAR = OFF_TINFO + TI * 16;
  static constexpr int NBAR = 2 * RING + 2 * NSQ + 2 * NAV + 2 + 2 * 2 + 2 * MR;
  static constexpr int OFF_RED = OFF_BAR + NBAR * 8;
  // softmax scratch per warpgroup: the flush's sums [4 warps][GH][NG + 1], then the tile maxima [4][GH + 1]
  static constexpr int RED_FLUSH = 4 * GH * (NG + 1);
  static constexpr int RED_GROUP = RED_FLUSH + 4 * (GH + 1);
  static constexpr int OFF_MISC = OFF_RED + ((SG * RED_GROUP * 4 + 15) / 16) * 16;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + slack to align the base to 1024
  static_assert(OFF_BQ % 1024 == 0 && OFF_BW % 1024 == 0 && BW_BYTES % 1024 == 0, "operand alignment");
  static_assert(STAGE_BYTES % 16 == 0 && OFF_RING % 16 == 0, "bulk copy alignment");
  static_assert(TM_USED <= 512 && GH * NG * 2 <= NCG && (!QK8 || GH * NG * QT <= NQG), "tensor memory and columns");
  static_assert(!BW_MN || (GH * NG * 2 == NCG && NCG % 8 == 0), "MN-major weights: every column of a 16-byte chunk written");
  static_assert(!QKG || (2 * G * NG == N && 2 * G % 16 == 0 && 2 * GH % 8 == 0 && NQG == 2 * GH * NG), "per-group Q.K");
  static_assert(SMEM <= 232448, "shared memory per block");
};
// Column (and Q.K image row) of (head h, group g, term t): warpgroup h / GH owns the block of NCG columns
// starting at (h / GH) * NCG.
template <int G, int NG>
__host__ __device__ constexpr int col_of(int h, int g, int t) {
  using C = Cfg<G, NG>;
  return (h / C::GH) * C::NCG + ((h % C::GH) * NG + g) * 2 + t;
}

// Tile information written by the producer (one 16-byte entry per tile).
struct TileInfo {
  int seg;                // b * Hkv + kvh
  int16_t ntok0, ntok1;   // valid tokens of page slots 0 and 1
  int flags;              // F_FIRST: first tile of a segment; F_LAST_SEG: last of a segment; F_LAST: last of the CTA
  int pad;
};
constexpr int F_FIRST = 1, F_LAST_SEG = 2, F_LAST = 4;

struct HArgs {
  PoolArgs p;
  const uint8_t *bq;  // per segment: Q.K operand image and score factors (qrot_kernel), BQ_BYTES apart
  float *part;        // partial slots [*][G][PART_STRIDE]
  int n_hist;
};

// Barriers (offsets in uint64 units from OFF_BAR).
template <int G, int NG>
struct Bars {
  uint64_t *full, *empty;          // [RING]   page stage landed / released (8 unpack warps)
  uint64_t *ak_full, *qk_done;     // [NSQ]    K codes in TMEM (4 warps) / the tile's Q.K done: S ready and the
                                   //          K buffer free (MMA commit)
  uint64_t *av_full, *pv_done;     // [NAV]    V tile in smem (4 warps) / the tile's P.V done: the V tile, the
                                   //          weight buffer and the accumulator free (MMA commit)
  uint64_t *w_full;                // [2]      weights of a tile written (4 warps per softmax warpgroup)
  uint64_t *bq_full, *bq_free;     // [2]      Q.K operand image landed / released (MMA commit + softmax warps)
  uint64_t *meta_full, *meta_free; // [MR]     scale/zero of a tile copied (4 K-unpack warps) / read (softmax)
  __device__ Bars(uint8_t *sm) {
    uint64_t *b = reinterpret_cast<uint64_t *>(sm + Cfg<G, NG>::OFF_BAR);
    constexpr int R = Cfg<G, NG>::RING, NV = Cfg<G, NG>::NAV;
    full = b; empty = b + R;
    constexpr int NS = Cfg<G, NG>::NSQ;
    ak_full = b + 2 * R; qk_done = ak_full + NS;
    av_full = qk_done + NS; pv_done = av_full + NV;
    w_full = pv_done + NV;
    bq_full = w_full + 2; bq_free = bq_full + 2;
    meta_full = bq_free + 2; meta_free = meta_full + MR;
  }
};

constexpr int M_TMEM = 0, M_ABORT = 1;

__device__ __forceinline__ bool aborted(const uint32_t *misc) {
  return *reinterpret_cast<const volatile uint32_t *>(misc + M_ABORT) != 0;
}
__device__ __noinline__ void set_abort(const PoolArgs &p, uint32_t *misc) {
  *reinterpret_cast<volatile uint32_t *>(misc + M_ABORT) = 1;
  atomicOr(p.err, OSCAR_DEVERR_TIMEOUT);
}
// Bounded wait (one second); on timeout the CTA's abort flag and the pool's timeout bit are set.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, const PoolArgs &p, uint32_t *misc) {
  if (mbar_try_wait_hint(bar, parity, 1000000u)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_hint(bar, parity, 1000000u)) {
    if (aborted(misc)) return false;
    if (globaltimer_ns() - t0 > 1000000000ull) {
      set_abort(p, misc);
      return false;
    }
  }
  return true;
}
// Warp-collective bounded wait: every lane polls the barrier (no divergence); true on every lane when the phase
// completed.  A completed phase stays completed for try_wait, so the vote settles after one more poll.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const PoolArgs &p, uint32_t *misc) {
  if (__all_sync(FULL, mbar_try_wait_hint(bar, parity, 1000000u))) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!__all_sync(FULL, mbar_try_wait_hint(bar, parity, 1000000u))) {
    if (__any_sync(FULL, aborted(misc))) return false;
    if (globaltimer_ns() - t0 > 1000000000ull) {
      if ((threadIdx.x & 31) == 0) set_abort(p, misc);
      return false;
    }
  }
  return true;
}

// ---- tcgen05 helpers (kind::f16, A from tensor memory or shared memory) ----
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major = false) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// 128-byte-swizzled operand descriptor with explicit leading / stride byte offsets.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
               ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// kind::f8f6f4 with A from tensor memory (both operands e4m3: instruction-descriptor format fields 0).
__device__ __forceinline__ void mma_tmem_a_f8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n"
               ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_smem_a(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
// N (a multiple of 8) consecutive fp32 columns of this warp's 32 TMEM lanes, in chunks of 8.
// Loads issued without waiting (tcgen05_wait_ld() before the registers are used).
template <int N>
__device__ __forceinline__ void tmem_ld_cols_async(uint32_t taddr, uint32_t *r) {
  static_assert(N % 8 == 0, "columns in chunks of 8");
#pragma unroll
  for (int c = 0; c < N; c += 8)
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[c + 0]), "=r"(r[c + 1]), "=r"(r[c + 2]), "=r"(r[c + 3]), "=r"(r[c + 4]), "=r"(r[c + 5]),
                   "=r"(r[c + 6]), "=r"(r[c + 7])
                 : "r"(taddr + c));
}
__device__ __forceinline__ void tcgen05_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  uint32_t r[N];
  tmem_ld_cols_async<N>(taddr, r);
  tcgen05_wait_ld();
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[N]) {
  static_assert(N % 8 == 0, "columns in chunks of 8");
#pragma unroll
  for (int c = 0; c < N; c += 8)
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr + c),
                 "r"(__float_as_uint(v[c + 0])), "r"(__float_as_uint(v[c + 1])), "r"(__float_as_uint(v[c + 2])),
                 "r"(__float_as_uint(v[c + 3])), "r"(__float_as_uint(v[c + 4])), "r"(__float_as_uint(v[c + 5])),
                 "r"(__float_as_uint(v[c + 6])), "r"(__float_as_uint(v[c + 7]))
                 : "memory");
  tmem_wait_st();
}

// Unpack one 32-bit word of 16 codes (code j at bits 2j) into 8 fp16x2 registers r[0..7]: register k holds
// codes (k, 8 + k) as the subnormals c * 4^k' * 2^-24, k' = k (k <= 4) or k - 5 (k >= 5).  Channel position
// p = 16 w + 2 k + half (w the word) of the operand holds channel 16 w + k + 8 half.
__device__ __forceinline__ void unpack_word(uint32_t x, uint32_t *r) {
#pragma unroll
  for (int k = 0; k < 5; ++k) r[k] = x & (0x00030003u << (2 * k));
  const uint32_t xs = x >> 10;
#pragma unroll
  for (int k = 0; k < 3; ++k) r[5 + k] = xs & (0x00030003u << (2 * k));
}
// The same word as e4m3 subnormals for the fp8 Q.K: register i (0..3) byte b holds code 4 b + i, as c * 2^-9
// (i even: the code in the mantissa's low bits) or c * 2^-7 (i odd: two bits up, the exponent's low bit taking
// the code's high bit: 1 -> 2^-7, 2 -> 2^-6, 3 -> 1.5 * 2^-6, linear in c).  Operand position p = 16 w + 4 i + b
// (w the word) holds channel 16 w + 4 b + i.
__device__ __forceinline__ void unpack_word_f8(uint32_t x, uint32_t *r) {
  r[0] = x & 0x03030303u;
  r[1] = x & 0x0C0C0C0Cu;
  const uint32_t xs = x >> 4;
  r[2] = xs & 0x03030303u;
  r[3] = xs & 0x0C0C0C0Cu;
}
__host__ __device__ __forceinline__ int pos8_channel(int p) { return (p & ~15) + 4 * (p & 3) + ((p & 15) >> 2); }
__host__ __device__ __forceinline__ bool pos8_low(int p) { return ((p >> 2) & 1) == 0; }  // code factor 2^-9
__host__ __device__ __forceinline__ int pos_channel(int p) { return (p & ~15) + ((p & 15) >> 1) + 8 * (p & 1); }
__host__ __device__ __forceinline__ int pos_k(int p) {
  const int k = (p & 15) >> 1;
  return k <= 4 ? k : k - 5;
}
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }
// Byte offset of 16-bit element (row, k) (k < 128) of a [rows][128] K-major operand stored as two 128-byte-
// swizzled atom columns of `rows` rows each.
__host__ __device__ __forceinline__ int op_offset(int rows, int row, int k) {
  return (k >> 6) * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
         (k & 7) * 2;
}

// ---------------------------------------------------------------------------------------------
// Query rotation and the Q.K operand image of one (sequence, KV head): grid B * Hkv, 512 threads.
// Image rows n = (h * NG + g) * 2 + term (term 0: hi, 1: lo), K position p -> channel pos_channel(p):
// the term of y = q_rot[h][ch] * 2^sigma_h times 4^-pos_k(p) when ch lies in group g, else 0.  Factors:
// kf[h] = 2^(24 - sigma_h) log2(e) s, zf[h][g] = sum over the group of q_rot[h][ch] * log2(e) s.
// Loads of q and R_k come before griddepcontrol.wait; the trigger follows it (the history kernel reads the
// pool counters at once, so it must start after the previous step's merge has completed).
template <int G, int NG>
__global__ void __launch_bounds__(256) qrot_kernel(PoolArgs p, const uint16_t *q, uint8_t *bq, float sm_log2) {
  using C = Cfg<G, NG>;
  __shared__ float qs[G][D];
  __shared__ float part2[2][G][D];
  __shared__ int s_sig[G];
  const int s = blockIdx.x, b = s / p.Hkv, kvh = s % p.Hkv;
  const int tid = threadIdx.x, c = tid & (D - 1), half = tid >> 7;
  // thread (c, half) sums rows 64 half .. 64 half + 63 of column c; all 64 loads are issued at once, before
  // the wait for the previous kernel (R_k is not written by the decode)
  const float *R = p.R_k + (size_t)kvh * D * D + (size_t)(64 * half) * D + c;
  float r[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) r[i] = R[(size_t)i * D];
  for (int i = tid; i < G * D; i += 256) qs[i / D][i % D] = bf16_to_f32(q[((size_t)b * p.Hq + kvh * G) * D + i]);
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i)
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = fmaf(qs[h][64 * half + i], r[i], acc[h]);
#pragma unroll
  for (int h = 0; h < G; ++h) part2[half][h][c] = acc[h];
  __syncthreads();
  if (half == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) qs[h][c] = part2[0][h][c] + part2[1][h][c];
  __syncthreads();
  if (!OSCAR_DCHECK(s < p.B * p.Hkv, p.err)) return;
  uint8_t *img = bq + (size_t)s * C::BQ_BYTES;
  float *fac = reinterpret_cast<float *>(img + C::BQ_IMG);
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < G) {
    const int h = warp;
    float amax = 0.f;
    float gs[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) gs[g] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int ch = lane + 32 * k;
      const float v = qs[h][ch];
      amax = fmaxf(amax, fabsf(v));
#pragma unroll
      for (int g = 0; g < NG; ++g)
        if (ch / (D / NG) == g) gs[g] += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, o));
#pragma unroll
      for (int g = 0; g < NG; ++g) gs[g] += __shfl_xor_sync(FULL, gs[g], o);
    }
    if (lane == 0) {
      int e = 0;
      if (amax > 0.f) frexpf(amax, &e);
      const int sig = (amax > 0.f) ? 14 - e : 0;  // amax * 2^sig < 2^14
      s_sig[h] = sig;
      // score factor: sum_c code_c q_rot_c = 2^(24 - sigma) (S_hi + S_lo) (fp16 split), or 2^(-2 - sigma)
      // sum_t 16^t S_t (fp8 digits)
      fac[h] = pow2i(C::QK8 ? -2 - sig : 24 - sig) * sm_log2;
#pragma unroll
      for (int g = 0; g < NG; ++g) fac[G + h * NG + g] = gs[g] * sm_log2;
    }
  }
  __syncthreads();
  if constexpr (C::QK8) {
    // the fp8 image: NQ rows x 128 e4m3 (one 128-byte-swizzled atom column); row sg * NQG + (hl * NG + g) * 6 + t
    // holds digit t of Y = rint(q_rot[h][ch] * 2^sigma * 2^9) (|Y| < 2^23) in balanced base 16,
    // Y = sum_t 16^t d_t with |d_t| <= 8, times 4 where the code of position p sits two bits lower
    // (code factor 2^-9 instead of 2^-7): every product is c * d * 2^-7 and a column's 128 sum exactly.
    for (int i = tid; i < C::NQ * (D / 4); i += 256) {
      const int n = i / (D / 4), p4 = 4 * (i % (D / 4));
      const int sgi = n / C::NQG, loc = n % C::NQG;
      uint32_t word = 0;
      if (sgi < C::SG && loc < C::GH * NG * C::QT) {
        const int h = sgi * C::GH + loc / (NG * C::QT), g = (loc / C::QT) % NG, t = loc % C::QT;
        const float s2 = pow2i(s_sig[h] + 9);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pp = p4 + e, ch = pos8_channel(pp);
          float dv = 0.f;
          if (ch / (D / NG) == g) {
            int Y = __float2int_rn(qs[h][ch] * s2);
            int d = 0;
            for (int k = 0; k <= t; ++k) {
              d = (k == C::QT - 1) ? Y : ((Y + 8) & 15) - 8;
              Y = (Y - d) >> 4;  // exact: Y - d is a multiple of 16
            }
            dv = (float)(pos8_low(pp) ? 4 * d : d);
          }
          const __nv_fp8_e4m3 f8(dv);  // exact: |dv| <= 32 with at most four significant bits
          word |= (uint32_t)f8.__x << (8 * e);
        }
      }
      *reinterpret_cast<uint32_t *>(img + (n >> 3) * 1024 + (n & 7) * 128 + ((((p4 >> 4) ^ (n & 7))) << 4) +
                                    (p4 & 15)) = word;
    }
  } else {
    // the fp16 image: N rows x 128 positions, two 16-bit values per thread-step
    for (int i = tid; i < C::N * (D / 2); i += 256) {
      const int n = i / (D / 2), p2 = 2 * (i % (D / 2));
      uint32_t word = 0;
      const int sgi = n / C::NCG, loc = n % C::NCG;  // row n = col_of(h, g, term), or g 2G + 2h + term (QKG)
      if (C::QKG || loc < C::GH * NG * 2) {
        const int h = C::QKG ? (n % (2 * G)) / 2 : sgi * C::GH + loc / (2 * NG);
        const int g = C::QKG ? n / (2 * G) : (loc / 2) % NG, term = n & 1;
        const float s2 = pow2i(s_sig[h]);
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pp = p2 + e, ch = pos_channel(pp);
          float t = 0.f;
          if (ch / (D / NG) == g) {
            const float y = qs[h][ch] * s2;  // exact: s2 is a power of two
            const float hi = 8.f * rintf(y * 0.125f);
            const float lo = rintf((y - hi) * 256.f) * (1.f / 256.f);
            t = (term == 0 ? hi : lo) * pow2i(-2 * pos_k(pp));
          }
          v[e] = t;
        }
        word = pack_half2(v[0], v[1]);
      }
      *reinterpret_cast<uint32_t *>(img + op_offset(C::N, n, p2)) = word;
    }
  }
}

// ---------------------------------------------------------------------------------------------
template <int G, int NG>
struct Smem {
  uint8_t *base;
  __device__ uint8_t *av(int i) const { return base + Cfg<G, NG>::OFF_AV + i * AV_BYTES; }
  __device__ uint8_t *bq(int i) const { return base + Cfg<G, NG>::OFF_BQ + i * Cfg<G, NG>::BQ_STRIDE; }
  __device__ uint8_t *bw(int i) const { return base + Cfg<G, NG>::OFF_BW + i * Cfg<G, NG>::BW_BYTES; }
  __device__ uint8_t *stage(int i) const { return base + Cfg<G, NG>::OFF_RING + i * Cfg<G, NG>::STAGE_BYTES; }
  __device__ uint8_t *mring(int i) const { return base + Cfg<G, NG>::OFF_MRING + i * Cfg<G, NG>::MRING_TILE; }
  __device__ TileInfo *tinfo(int j) const {
    return reinterpret_cast<TileInfo *>(base + Cfg<G, NG>::OFF_TINFO) + (j % TI);
  }
  __device__ float *red() const { return reinterpret_cast<float *>(base + Cfg<G, NG>::OFF_RED); }
  __device__ uint32_t *misc() const { return reinterpret_cast<uint32_t *>(base + Cfg<G, NG>::OFF_MISC); }
};

// ---------------------------------------------------------------------------------------------
template <int G, int NG>
__global__ void __maxnreg__((Cfg<G, NG>::MAXREG)) hist_kernel(HArgs a) {
  using C = Cfg<G, NG>;
  extern __shared__ uint8_t smem_raw[];
  Smem<G, NG> sm{smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u)};
  Bars<G, NG> bar(sm.base);
  uint32_t *misc = sm.misc();
  const PoolArgs &p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  // the BF16 kernel that follows may start at once: it runs beside this one (it reads nothing this writes)
  pdl_trigger();

  __shared__ long long s_lo, s_n;
  __shared__ int s_b0, s_kvh0, s_local0, s_np0, s_hl0;
  if (tid == 0) {
    for (int i = 0; i < C::RING; ++i) { mbar_init(bar.full + i, 1); mbar_init(bar.empty + i, 8); }
    for (int i = 0; i < C::NSQ; ++i) { mbar_init(bar.ak_full + i, 4); mbar_init(bar.qk_done + i, 1); }
    for (int i = 0; i < C::NAV; ++i) { mbar_init(bar.av_full + i, 4); mbar_init(bar.pv_done + i, 1); }
    for (int i = 0; i < MR; ++i) { mbar_init(bar.meta_full + i, 4); mbar_init(bar.meta_free + i, 4 * C::SG); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar.w_full + i, 4 * C::SG);
      mbar_init(bar.bq_full + i, 1); mbar_init(bar.bq_free + i, 1 + 4 * C::SG);
    }
    misc[M_ABORT] = 0;
    mbar_fence_init();
  }
  if (warp == W_PROD) {
    long long lo, n;
    int b0, kvh0, local0, np0, hl0;
    split::Plan pl;
    split::locate_range(p, a.n_hist, cta, false, lo, n, b0, kvh0, local0, np0, hl0, pl);
    if (lane == 0) { s_lo = lo; s_n = n; s_b0 = b0; s_kvh0 = kvh0; s_local0 = local0; s_np0 = np0; s_hl0 = hl0; }
  }
  if (warp == W_MMA) tmem_alloc(misc + M_TMEM, C::TM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[M_TMEM];
  const long long n_pages = s_n;

  if (n_pages > 0) {
    if (warp == W_PROD) {
      // ---------------- producer: pages and Q.K operand images ----------------
      const uint64_t stream_pol = l2_evict_first();
      int b = s_b0, kvh = s_kvh0, local = s_local0, np = s_np0, hl = s_hl0;
      long long done = 0;
      int j = 0, sigma = -1, cur_seg = -1, pt_base = -1, pt_b = -1, ptv = -1;
      bool waited = false;  // griddepcontrol.wait done (the images come from the query rotation)
      int pending = -1;     // segment whose image is still to be copied (before the wait)
      auto copy_image = [&](int sg, int sig) -> bool {
        constexpr int BQN = C::BQN;
        const int bi = sig % BQN;
        if (sig >= BQN && !warp_wait(bar.bq_free + bi, ((sig - BQN) / BQN) & 1, p, misc)) return false;
        if (lane == 0) {
          if (OSCAR_DCHECK(sg >= 0 && sg < p.B * p.Hkv, p.err)) {
            mbar_arrive_expect_tx(bar.bq_full + bi, (uint32_t)C::BQ_BYTES);
            bulk_g2s(sm.bq(bi), a.bq + (size_t)sg * C::BQ_BYTES, (uint32_t)C::BQ_BYTES, bar.bq_full + bi);
          } else {
            mbar_arrive(bar.bq_full + bi);
          }
        }
        return true;
      };
      bool ok = true;
      while (done < n_pages && ok) {
        const int stage = j % C::RING;
        if (j >= C::RING && !warp_wait(bar.empty + stage, ((j / C::RING) - 1) & 1, p, misc)) { ok = false; break; }
        const int seg = b * p.Hkv + kvh;
        const int cnt = (int)min(2ll, min(n_pages - done, (long long)(np - local)));
        if (cnt <= 0) {  // counters inconsistent with the range (changed during the launch): stop; the other
          if (lane == 0) atomicOr(p.err, OSCAR_DEVERR_COUNTERS);  // roles end at their bounded waits
          ok = false;
          break;
        }
        int flags = 0;
        const bool new_seg = seg != cur_seg;
        if (new_seg) {
          flags |= F_FIRST;
          ++sigma;
          cur_seg = seg;
        }
        if (local + cnt == np) flags |= F_LAST_SEG;
        if (done + cnt >= n_pages) flags |= F_LAST | F_LAST_SEG;
        // page-table entries, 32 at a time per sequence (lane i holds entry pt_base + i)
        if (b != pt_b || local < pt_base || local + cnt > pt_base + 32) {
          pt_b = b;
          pt_base = local;
          ptv = local + lane < np ? ld_hint(p.page_table + (size_t)b * p.max_pages + local + lane, l2_evict_last()) : -1;
        }
        int pp = __shfl_sync(FULL, ptv, (local - pt_base + lane) & 31);
        int ntk = 0;
        if (lane < cnt) {
          ntk = min(PAGE, hl - (local + lane) * PAGE);
          if (pp < 0 || pp >= p.num_pages) {
            atomicOr(p.err, OSCAR_DEVERR_PAGE_INDEX);
            pp = -1;
          }
        } else {
          pp = -1;
        }
        const bool have = pp >= 0;
        const unsigned hv = __ballot_sync(FULL, have);
        const int n0 = __shfl_sync(FULL, have ? ntk : 0, 0), n1 = __shfl_sync(FULL, have ? ntk : 0, 1);
        if (lane == 0) {
          TileInfo ti;
          ti.seg = seg; ti.ntok0 = (int16_t)n0; ti.ntok1 = (int16_t)n1; ti.flags = flags; ti.pad = 0;
          *sm.tinfo(j) = ti;
          mbar_arrive_expect_tx(bar.full + stage, (uint32_t)(__popc(hv & 3u) * C::PAGE_BYTES));
        }
        __syncwarp();
        if (lane < 2 && have) {
          uint8_t *dst = sm.stage(stage) + lane * C::PAGE_BYTES;
          const size_t row = ((size_t)pp * p.Hkv + kvh) * PAGE;
          const int mb = PAGE * C::META;
          bulk_g2s_hint(dst + OFF_KC, p.codes_k + row * (D / 4), 2048, bar.full + stage, stream_pol);
          bulk_g2s_hint(dst + OFF_VC, p.codes_v + row * (D / 4), 2048, bar.full + stage, stream_pol);
          bulk_g2s_hint(dst + OFF_META, p.scale_k + row * NG, mb, bar.full + stage, stream_pol);
          bulk_g2s_hint(dst + OFF_META + mb, p.zero_k + row * NG, mb, bar.full + stage, stream_pol);
          bulk_g2s_hint(dst + OFF_META + 2 * mb, p.scale_v + row * NG, mb, bar.full + stage, stream_pol);
          bulk_g2s_hint(dst + OFF_META + 3 * mb, p.zero_v + row * NG, mb, bar.full + stage, stream_pol);
        }
        done += cnt;
        local += cnt;
        ++j;
        if (local == np && done < n_pages) {
          local = 0;
          if (++kvh == p.Hkv) {
            kvh = 0;
            do { ++b; } while (b < p.B && ((max(0, min(split::hist_len_of(p, b), p.max_pages * PAGE)) + PAGE - 1) / PAGE) == 0);
            if (b < p.B) {
              hl = max(0, min(split::hist_len_of(p, b), p.max_pages * PAGE));
              np = (hl + PAGE - 1) / PAGE;
            }
          }
        }
        // A new segment's operand image is copied after its first tile's pages: with one image buffer the
        // copy waits for the previous segment's last Q.K, which the MMA thread issues only once it sees this
        // tile.  The first segment's image waits for the first ring of page copies (the query rotation that
        // writes it may still be running) or for the first segment change.
        if (new_seg) {
          if (sigma == 0) {
            pending = seg;
          } else {
            if (!waited) {
              pdl_wait();
              waited = true;
              if (pending >= 0 && !copy_image(pending, 0)) { ok = false; break; }
              pending = -1;
            }
            if (!copy_image(seg, sigma)) { ok = false; break; }
          }
        }
        if (ok && !waited && (j >= C::RING || done >= n_pages)) {
          pdl_wait();
          waited = true;
          if (pending >= 0 && !copy_image(pending, 0)) ok = false;
          pending = -1;
        }
      }
      if (!ok) {
        // copies still in flight must land before the CTA exits
        if (lane == 0)
          for (int k = max(0, j - C::RING); k < j; ++k)
            mbar_wait_bounded(bar.full + k % C::RING, (uint32_t)((k / C::RING) & 1), 100000000ull);
      }
    } else if (warp == W_MMA) {
      // ---------------- MMA issuer (one thread) ----------------
      // Q.K runs up to two tiles ahead of P.V (NSQ >= 3 S and K buffers), so that the tensor pipe has work
      // queued while the softmax of the current tile runs.  One commit per Q.K (qk_done: S ready, K buffer
      // free) and one per P.V (pv_done: V tile, weight buffer and accumulator released).
      if (lane == 0) {
        // the e4m3 formats of kind::f8f6f4 and the f16 formats of kind::f16 share the descriptor value 0
        constexpr uint32_t ID_QK = idesc_f16(TILE, C::NQ, false), ID_PV = idesc_f16(TILE, C::N, true, C::BW_MN);
        constexpr uint32_t ID_QKG = idesc_f16(TILE, 2 * G, false);
        constexpr int NS = C::NSQ;
        int sigma = -1, nq = 0, j = 0;
        int sig_of[NS];
        bool first_of[NS];
        bool more = true, ok = true;
        // issue Q.K of tile nq (its K codes in tensor memory; its segment's operand image in smem)
        auto issue_qk = [&]() -> bool {
          const int t = nq;
          if (!wait_bar(bar.ak_full + (t % NS), (t / NS) & 1, p, misc)) return false;
          tc_fence_after();
          const TileInfo ti = *sm.tinfo(t);
          if (ti.flags & F_FIRST) {
            if (sigma >= 0) umma_commit(bar.bq_free + (sigma % C::BQN));  // segment sigma's last Q.K is issued
            ++sigma;
            if (!wait_bar(bar.bq_full + (sigma % C::BQN), (sigma / C::BQN) & 1, p, misc)) return false;
            tc_fence_after();
          }
          sig_of[t % NS] = sigma;
          first_of[t % NS] = (ti.flags & F_FIRST) != 0;
          const uint32_t bq = smem_u32(sm.bq(sigma % C::BQN));
          const uint32_t d = tmem + C::TM_S + C::NQ * (t % NS), a = tmem + C::TM_AK + C::AKC * (t % NS);
          if constexpr (C::QK8) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K = 32 e4m3 per MMA: 32 bytes of the operand rows
              mma_tmem_a_f8(d, a + 8 * kk, desc_sw128(bq + kk * 32, 16, 1024), ID_QK, kk > 0 ? 1u : 0u);
          } else if constexpr (C::QKG) {
            constexpr int KPG = 8 / NG;  // 16-channel steps per group
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const int g = kk / KPG;
              mma_tmem_a(d + 2 * G * g, a + 8 * kk,
                         desc_sw128(bq + (kk >> 2) * (C::N * 128) + g * (2 * G / 8) * 1024 + (kk & 3) * 32, 16, 1024),
                         ID_QKG, (kk % KPG) > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_tmem_a(d, a + 8 * kk, desc_sw128(bq + (kk >> 2) * (C::N * 128) + (kk & 3) * 32, 16, 1024), ID_QK,
                         kk > 0 ? 1u : 0u);
          }
          umma_commit(bar.qk_done + (t % NS));
          if (ti.flags & F_LAST) more = false;
          ++nq;
          return true;
        };
        ok = issue_qk();
        if (ok && more) ok = issue_qk();
        while (ok) {
          if (more && !issue_qk()) break;  // tile j + 2
          if (!wait_bar(bar.w_full + (j & 1), (j >> 1) & 1, p, misc)) break;
          if (!wait_bar(bar.av_full + (j % C::NAV), (j / C::NAV) & 1, p, misc)) break;
          tc_fence_after();
          const uint32_t av = smem_u32(sm.av(j % C::NAV)), bw = smem_u32(sm.bw(j & 1));
          const uint32_t o = tmem + C::TM_O + C::N * (sig_of[j % NS] & 1);
          const bool first = first_of[j % NS];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_smem_a(o, desc_sw128(av + 2048 * kk, 16384, 1024),
                       C::BW_MN ? desc_sw128(bw + 2048 * kk, C::BW_BYTES, 1024)
                                : desc_sw128(bw + (kk >> 2) * (C::N * 128) + (kk & 3) * 32, 16, 1024),
                       ID_PV, (kk > 0 || !first) ? 1u : 0u);
          umma_commit(bar.pv_done + (j % C::NAV));
          if (!more && j == nq - 1) break;  // that was the CTA's last tile
          ++j;
        }
        // every MMA this thread issued completes before tensor memory is freed
        umma_commit(bar.bq_free + (max(sigma, 0) % C::BQN));
        mbar_wait_bounded(bar.pv_done + (j % C::NAV), (uint32_t)((j / C::NAV) & 1), 100000000ull);
      }
    } else if (warp < W_V0) {
      // ---------------- K codes -> tensor memory (A of Q.K); scale/zero -> the meta ring ----------------
      const int quad = warp & 3, t = 32 * quad + lane, slot = t >> 6, row = t & 63;
      const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
      for (int j = 0;; ++j) {
        const int stage = j % C::RING;
        if (!warp_wait(bar.full + stage, (j / C::RING) & 1, p, misc)) break;
        const TileInfo ti = *sm.tinfo(j);
        // the K operand buffer of tile j - NSQ and the meta-ring slot of tile j - MR are free
        if (j >= C::NSQ && !warp_wait(bar.qk_done + (j % C::NSQ), ((j / C::NSQ) - 1) & 1, p, misc)) break;
        if (j >= MR && !warp_wait(bar.meta_free + (j % MR), ((j / MR) - 1) & 1, p, misc)) break;
        const uint8_t *pg = sm.stage(stage) + slot * C::PAGE_BYTES;
        const uint4 c0 = *reinterpret_cast<const uint4 *>(pg + OFF_KC + row * 32);
        const uint4 c1 = *reinterpret_cast<const uint4 *>(pg + OFF_KC + row * 32 + 16);
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        tc_fence_after();
        if constexpr (C::QK8) {
          uint32_t r[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) unpack_word_f8(w[i], r + 4 * i);
          tmem_st32(tmem + lane_addr + C::TM_AK + C::AKC * (j % C::NSQ), r);
        } else {
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {  // two stores of 32 columns (register pressure)
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) unpack_word(w[4 * hlf + i], r + 8 * i);
            tmem_st32(tmem + lane_addr + C::TM_AK + C::AKC * (j % C::NSQ) + 32 * hlf, r);
          }
        }
        // scale/zero of the token: Ks, Kz, Vs, Vz (NG bf16 each) -> one record of the meta ring
        {
          uint8_t *mr = sm.mring(j % MR) + t * 4 * C::META;
          const uint8_t *mp = pg + OFF_META + row * C::META;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if constexpr (NG == 1) {
              *reinterpret_cast<uint16_t *>(mr + 2 * q) = *reinterpret_cast<const uint16_t *>(mp + q * PAGE * C::META);
            } else if constexpr (NG == 2) {
              *reinterpret_cast<uint32_t *>(mr + 4 * q) = *reinterpret_cast<const uint32_t *>(mp + q * PAGE * C::META);
            } else {
              *reinterpret_cast<uint2 *>(mr + 8 * q) = *reinterpret_cast<const uint2 *>(mp + q * PAGE * C::META);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar.ak_full + (j % C::NSQ));
          mbar_arrive(bar.meta_full + (j % MR));
          mbar_arrive(bar.empty + stage);
        }
        if (ti.flags & F_LAST) break;
      }
    } else if (warp < W_S0) {
      // ---------------- V codes -> the swizzled shared-memory tile (A of P.V, MN-major) ----------------
      const int t = 32 * (warp - W_V0) + lane, slot = t >> 6, row = t & 63;
      uint32_t choff[8];  // swizzled 16-byte chunk c of the token's 128-byte atom row
#pragma unroll
      for (int c = 0; c < 8; ++c) choff[c] = (uint32_t)(((c ^ (t & 7)) << 4) + (t >> 3) * 1024 + (t & 7) * 128);
      for (int j = 0;; ++j) {
        const int stage = j % C::RING;
        if (!warp_wait(bar.full + stage, (j / C::RING) & 1, p, misc)) break;
        const TileInfo ti = *sm.tinfo(j);
        // P.V of tile j - NAV has completed: its V tile buffer is free
        if (j >= C::NAV && !warp_wait(bar.pv_done + (j % C::NAV), ((j / C::NAV) - 1) & 1, p, misc)) break;
        const uint8_t *pg = sm.stage(stage) + slot * C::PAGE_BYTES;
        const uint4 c0 = *reinterpret_cast<const uint4 *>(pg + OFF_VC + row * 32);
        const uint4 c1 = *reinterpret_cast<const uint4 *>(pg + OFF_VC + row * 32 + 16);
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint8_t *av = sm.av(j % C::NAV);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t r[8];
          unpack_word(w[i], r);
          // registers r[0..3] -> 16-byte chunk c = 2 i, r[4..7] -> chunk 2 i + 1 of the token's 256-byte row
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            const int c = 2 * i + hlf;
            *reinterpret_cast<uint4 *>(av + (c >> 3) * 16384 + choff[c & 7]) =
                make_uint4(r[4 * hlf], r[4 * hlf + 1], r[4 * hlf + 2], r[4 * hlf + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar.av_full + (j % C::NAV));
          mbar_arrive(bar.empty + stage);
        }
        if (ti.flags & F_LAST) break;
      }
    } else {
      // ---------------- softmax warpgroup sg: heads [sg GH, sg GH + GH) of every tile ----------------
      // (thread = token row of S, channel row of O)
      constexpr int GH = C::GH, NCG = C::NCG;
      const int sg = (warp - W_S0) >> 2, quad = warp & 3, r = 32 * quad + lane, sw = (warp - W_S0) & 3;
      const int nbar = 1 + sg;  // named barrier of the warpgroup
      const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
      const int cbase = sg * NCG;  // this warpgroup's columns of S and O
      float mref[GH], lpart[GH], ozp[GH][NG], kf[GH], zf[GH][NG];
      int tau = 0;
      float tau_lim = 0.f;
      int sigma = -1, seg = -1, prev_tile = -1;  // prev_tile: last tile of the current segment so far
      float *red = sm.red() + sg * C::RED_GROUP;
      const int pch = pos_channel(r), pgrp = pch / (D / NG), pk = pos_k(r);
      // byte offset of (row cbase + n, token r) in the weight operand: op_offset(N, cbase + n, r) split into a
      // per-thread part and, for the compile-time n of the unrolled loops, a row part; cbase is a multiple of 8
      const int bw_tok = (r >> 6) * C::N * 128 + (cbase >> 3) * 1024 + (r & 7) * 2, rcx = (r & 63) >> 3;
      auto bw_row = [rcx](int n) { return (n >> 3) * 1024 + (n & 7) * 128 + (((rcx ^ (n & 7))) << 4); };
      // Flush the segment's accumulator (after its last P.V) into partial slot (cta + seg), this
      // warpgroup's heads.
      auto flush = [&](int last_tile) -> bool {
        if (!warp_wait(bar.pv_done + (last_tile % C::NAV), (last_tile / C::NAV) & 1, p, misc)) return false;
        tc_fence_after();
        float o[NCG];
        tmem_ld_cols<NCG>(tmem + lane_addr + C::TM_O + C::N * (sigma & 1) + cbase, o);
        // l and the zero-point sums over the 128 rows: warp sums, then the four warps through shared memory
        float ls[GH], zs[GH][NG];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          ls[h] = lpart[h];
#pragma unroll
          for (int g = 0; g < NG; ++g) zs[h][g] = ozp[h][g];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int h = 0; h < GH; ++h) {
            ls[h] += __shfl_xor_sync(FULL, ls[h], off);
#pragma unroll
            for (int g = 0; g < NG; ++g) zs[h][g] += __shfl_xor_sync(FULL, zs[h][g], off);
          }
        named_bar_sync(nbar, 128);  // the previous use of red[] is over
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < GH; ++h) {
            red[(sw * GH + h) * (NG + 1)] = ls[h];
#pragma unroll
            for (int g = 0; g < NG; ++g) red[(sw * GH + h) * (NG + 1) + 1 + g] = zs[h][g];
          }
        }
        named_bar_sync(nbar, 128);
        // (the debug build checks the slot against the workspace's history slots: n_hist + B * Hkv)
        if (!OSCAR_DCHECK(cta + seg < a.n_hist + p.B * p.Hkv && seg >= 0, p.err)) return true;
        float *slot = a.part + ((size_t)cta + seg) * G * PART_STRIDE;
        const float unit = pow2i(24 - 2 * pk - tau);
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          float L = 0.f, Z = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            L += red[(w * GH + h) * (NG + 1)];
            Z += red[(w * GH + h) * (NG + 1) + 1 + pgrp];
          }
          const int c0 = (h * NG + pgrp) * 2, hg = sg * GH + h;
          slot[hg * PART_STRIDE + pch] = (o[c0] + o[c0 + 1]) * unit + Z;
          if (r == 0) {
            slot[hg * PART_STRIDE + D] = mref[h];
            slot[hg * PART_STRIDE + D + 1] = L;
          }
        }
        return true;
      };
      bool ok = true;
      for (int j = 0;; ++j) {
        // the K unpack of tile j has copied its scale/zero rows into the meta ring
        if (!warp_wait(bar.meta_full + (j % MR), (j / MR) & 1, p, misc)) { ok = false; break; }
        const TileInfo ti = *sm.tinfo(j);
        if (ti.flags & F_FIRST) {
          if (sigma >= 0 && !flush(prev_tile)) { ok = false; break; }
          ++sigma;
          seg = ti.seg;
          if (!warp_wait(bar.bq_full + (sigma % C::BQN), (sigma / C::BQN) & 1, p, misc)) { ok = false; break; }
          const float *fac = reinterpret_cast<const float *>(sm.bq(sigma % C::BQN) + C::BQ_IMG);
#pragma unroll
          for (int h = 0; h < GH; ++h) {
            kf[h] = fac[sg * GH + h];
            mref[h] = -INFINITY;
            lpart[h] = 0.f;
#pragma unroll
            for (int g = 0; g < NG; ++g) { zf[h][g] = fac[G + (sg * GH + h) * NG + g]; ozp[h][g] = 0.f; }
          }
          tau = 0;
          tau_lim = 0.f;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar.bq_free + (sigma % C::BQN));
          prev_tile = -1;
        }
        // scale/zero of this thread's token
        float ks[NG], kz[NG], vs[NG], vz[NG];
        {
          // the token's record: Ks[NG] Kz[NG] Vs[NG] Vz[NG] bf16, 8 NG bytes, read in 8- or 16-byte pieces
          uint32_t wd[2 * NG];
          const uint8_t *mr = sm.mring(j % MR) + r * 4 * C::META;
          if constexpr (NG == 1) {
            const uint2 v = *reinterpret_cast<const uint2 *>(mr);
            wd[0] = v.x; wd[1] = v.y;
          } else {
#pragma unroll
            for (int i = 0; i < NG / 2; ++i) {
              const uint4 v = reinterpret_cast<const uint4 *>(mr)[i];
              wd[4 * i] = v.x; wd[4 * i + 1] = v.y; wd[4 * i + 2] = v.z; wd[4 * i + 3] = v.w;
            }
          }
          auto half_at = [&](int idx) {  // bf16 number idx of the record
            return __uint_as_float((idx & 1) ? (wd[idx >> 1] & 0xffff0000u) : (wd[idx >> 1] << 16));
          };
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            ks[g] = half_at(g);
            kz[g] = half_at(NG + g);
            vs[g] = half_at(2 * NG + g);
            vz[g] = half_at(3 * NG + g);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.meta_free + (j % MR));
        const bool valid = r < 64 ? r < ti.ntok0 : (r - 64) < ti.ntok1;
        if (!valid) {
#pragma unroll
          for (int g = 0; g < NG; ++g) { vs[g] = 0.f; vz[g] = 0.f; }
        }
        if (!warp_wait(bar.qk_done + (j % C::NSQ), (j / C::NSQ) & 1, p, misc)) { ok = false; break; }
        tc_fence_after();
        constexpr int NQG = C::NQG;
        float s[NQG];
        if constexpr (C::QKG) {  // group g's columns of this warpgroup's heads: g 2G + 2 (sg GH) ...
          uint32_t sr[NQG];
#pragma unroll
          for (int g = 0; g < NG; ++g)
            tmem_ld_cols_async<2 * GH>(tmem + lane_addr + C::TM_S + C::NQ * (j % C::NSQ) + 2 * G * g + 2 * GH * sg,
                                       sr + 2 * GH * g);
          tcgen05_wait_ld();
#pragma unroll
          for (int c = 0; c < NQG; ++c) s[c] = __uint_as_float(sr[c]);
        } else {
          tmem_ld_cols<NQG>(tmem + lane_addr + C::TM_S + C::NQ * (j % C::NSQ) + sg * NQG, s);
        }
        float sc[GH];
        auto code_sum = [&](int h, int g) {  // head h's code sum of group g
          if constexpr (C::QK8) {  // sum_t 16^t S_t by Horner (exact until the last two steps)
            const float *st = s + (h * NG + g) * C::QT;
            float sum = st[C::QT - 1];
#pragma unroll
            for (int t = C::QT - 2; t >= 0; --t) sum = fmaf(sum, 16.f, st[t]);
            return sum;
          } else if constexpr (C::QKG) {
            return s[2 * GH * g + 2 * h] + s[2 * GH * g + 2 * h + 1];
          } else {
            return s[(h * NG + g) * 2] + s[(h * NG + g) * 2 + 1];
          }
        };
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          float acc, zacc;
          if constexpr (NG % 2 == 0) {  // groups in pairs: paired float32 products and sums
            float2 a2 = make_float2(0.f, 0.f), z2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int g = 0; g < NG; g += 2) {
              a2 = ffma2(make_float2(code_sum(h, g), code_sum(h, g + 1)), make_float2(ks[g], ks[g + 1]), a2);
              z2 = ffma2(make_float2(kz[g], kz[g + 1]), make_float2(zf[h][g], zf[h][g + 1]), z2);
            }
            acc = a2.x + a2.y;
            zacc = z2.x + z2.y;
          } else {
            acc = 0.f;
            zacc = 0.f;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              acc = fmaf(code_sum(h, g), ks[g], acc);
              zacc = fmaf(kz[g], zf[h][g], zacc);
            }
          }
          sc[h] = valid ? fmaf(acc, kf[h], zacc) : -INFINITY;
        }
        // reference and weight-scale updates, decided by the warpgroup's 128 threads together
        float vmax = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g) vmax = fmaxf(vmax, vs[g]);
        bool need = vmax > 0.f && vmax >= tau_lim;
#pragma unroll
        for (int h = 0; h < GH; ++h) need |= sc[h] > mref[h] + (float)LAZY;
        const bool any = !named_bar_and(nbar, 128, !need);
        if (any) {
          // maxima over the tile: warp reduction, then the four warps through shared memory
          float tm[GH];
#pragma unroll
          for (int h = 0; h < GH; ++h) tm[h] = sc[h];
          float vm = vmax;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int h = 0; h < GH; ++h) tm[h] = fmaxf(tm[h], __shfl_xor_sync(FULL, tm[h], off));
            vm = fmaxf(vm, __shfl_xor_sync(FULL, vm, off));
          }
          float *rr = red + C::RED_FLUSH;  // a region of its own (the flush's sums live below)
          if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GH; ++h) rr[sw * (GH + 1) + h] = tm[h];
            rr[sw * (GH + 1) + GH] = vm;
          }
          named_bar_sync(nbar, 128);
          float nm[GH], alpha[GH];
#pragma unroll
          for (int h = 0; h < GH; ++h)
            nm[h] = fmaxf(fmaxf(rr[h], rr[(GH + 1) + h]), fmaxf(rr[2 * (GH + 1) + h], rr[3 * (GH + 1) + h]));
          vm = fmaxf(fmaxf(rr[GH], rr[(GH + 1) + GH]), fmaxf(rr[2 * (GH + 1) + GH], rr[3 * (GH + 1) + GH]));
          named_bar_sync(nbar, 128);  // everyone has read rr[]
          int tnew = tau;
          if (vm > 0.f && vm >= tau_lim) {
            int e;
            frexpf(vm, &e);
            tnew = max(-100, min(100, WEXP - e - TAU_HEAD));
            if (tau_lim > 0.f && tnew > tau) tnew = tau;  // the scale only ever shrinks within a segment
          }
          bool rescale = false;
#pragma unroll
          for (int h = 0; h < GH; ++h) {
            const float m_new = nm[h] > mref[h] + (float)LAZY ? nm[h] : mref[h];
            alpha[h] = (mref[h] == -INFINITY || m_new == mref[h]) ? 1.f : exp2f(mref[h] - m_new);
            rescale |= alpha[h] != 1.f;
            mref[h] = m_new;
            lpart[h] *= alpha[h];
#pragma unroll
            for (int g = 0; g < NG; ++g) ozp[h][g] *= alpha[h];
          }
          const float tf = pow2i(tnew - tau);
          rescale |= (tau_lim > 0.f && tnew != tau);
          if (prev_tile >= 0 && rescale) {
            // the accumulator holds the earlier tiles of this segment: rescale this warpgroup's columns in
            // place once the last P.V into it has completed
            if (!warp_wait(bar.pv_done + (prev_tile % C::NAV), (prev_tile / C::NAV) & 1, p, misc)) { ok = false; break; }
            tc_fence_after();
            float o[NCG];
            const uint32_t oa = tmem + lane_addr + C::TM_O + C::N * (sigma & 1) + cbase;
            tmem_ld_cols<NCG>(oa, o);
#pragma unroll
            for (int h = 0; h < GH; ++h)
#pragma unroll
              for (int c = 0; c < 2 * NG; ++c) o[h * 2 * NG + c] *= alpha[h] * tf;
            tmem_st_cols<NCG>(oa, o);
          }
          if (tau_lim == 0.f || tnew != tau) {
            tau = tnew;
            tau_lim = pow2i(WEXP - tau);
          }
        }
        // weights (fp16 hi + lo) -> the B operand of P.V, token r of its K dimension
        // P.V of tile j - 2 has completed: the weight buffer of tile j is free
        if (j >= 2 && !warp_wait(bar.pv_done + ((j - 2) % C::NAV), ((j - 2) / C::NAV) & 1, p, misc)) { ok = false; break; }
        const float ut = pow2i(tau);
        float vsu[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) vsu[g] = vs[g] * ut;
        uint32_t wp[GH * NG];  // (hi, lo) of head h, group g as one fp16x2: columns (h NG + g) 2 and + 1
        auto split = [](float w) {  // w to 11 significant bits (hi) and the rest (lo), one packed conversion
          const float hi = __uint_as_float(__float_as_uint(w) & 0xffffe000u);
          const __half2 hl = __floats2half2_rn(hi, w - hi);
          return *reinterpret_cast<const uint32_t *>(&hl);
        };
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          const float pr = sc[h] == -INFINITY ? 0.f : fast_exp2(sc[h] - mref[h]);  // 0 past the tile's tokens
          lpart[h] += pr;
          if constexpr (NG % 2 == 0) {  // groups in pairs: paired float32 products, sums and hi/lo splits
#pragma unroll
            for (int g = 0; g < NG; g += 2) {
              const float2 prp = make_float2(pr, pr);
              const float2 oz = ffma2(prp, make_float2(vz[g], vz[g + 1]), make_float2(ozp[h][g], ozp[h][g + 1]));
              ozp[h][g] = oz.x;
              ozp[h][g + 1] = oz.y;
              const float2 w = fmul2(prp, make_float2(vsu[g], vsu[g + 1]));
              const float2 hi = make_float2(__uint_as_float(__float_as_uint(w.x) & 0xffffe000u),
                                            __uint_as_float(__float_as_uint(w.y) & 0xffffe000u));
              const float2 lo = fsub2(w, hi);
              const __half2 h0 = __floats2half2_rn(hi.x, lo.x), h1 = __floats2half2_rn(hi.y, lo.y);
              wp[h * NG + g] = *reinterpret_cast<const uint32_t *>(&h0);
              wp[h * NG + g + 1] = *reinterpret_cast<const uint32_t *>(&h1);
            }
          } else {
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              ozp[h][g] = fmaf(pr, vz[g], ozp[h][g]);
              wp[h * NG + g] = split(pr * vsu[g]);
            }
          }
        }
        if constexpr (C::BW_MN) {
          // row r of the tile: 16-byte chunk c (columns 8c .. 8c + 7) at ((c ^ (r & 7)) << 4)
          uint8_t *row = sm.bw(j & 1) + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int q = 0; q < GH * NG / 4; ++q) {
            const int c = (cbase >> 3) + q;
            *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) =
                make_uint4(wp[4 * q], wp[4 * q + 1], wp[4 * q + 2], wp[4 * q + 3]);
          }
        } else {
          uint8_t *bw = sm.bw(j & 1) + bw_tok;
#pragma unroll
          for (int i = 0; i < GH * NG; ++i) {
            *reinterpret_cast<uint16_t *>(bw + bw_row(2 * i)) = (uint16_t)(wp[i] & 0xffffu);
            *reinterpret_cast<uint16_t *>(bw + bw_row(2 * i + 1)) = (uint16_t)(wp[i] >> 16);
          }
        }
        if constexpr (!C::BW_MN && GH * NG * 2 < NCG) {
          uint8_t *bw = sm.bw(j & 1) + bw_tok;
          if (j < 2)  // padding rows of the weight operand: zero (once per buffer)
#pragma unroll
            for (int n = GH * NG * 2; n < NCG; ++n) *reinterpret_cast<uint16_t *>(bw + bw_row(n)) = 0;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.w_full + (j & 1));
        prev_tile = j;
        if (ti.flags & F_LAST) break;
      }
      if (ok && sigma >= 0) flush(prev_tile);
    }
  }
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
  // every thread has waited for the query rotation before the grid completes: the merge's wait (and the
  // next step's query rotation, which overwrites the operand images) follow it as well
  pdl_wait();
}

// ---------------------------------------------------------------------------------------------
// BF16 sink/window partials and (decode step) the demotion: 5 CTAs of 128 threads per (sequence, KV head).
struct BArgs {
  PoolArgs p;
  const uint16_t *q;
  float sm_log2;
  int n_hist;
  float *part;
  int step;
  const uint16_t *k_new, *v_new;
};
template <int G>
struct BSmem {
  part::BfSmem<G> bf;
  alignas(16) uint8_t scratch[part::DEMOTE_SCRATCH];
  alignas(16) float qrot[G][D];
};
static_assert(offsetof(BSmem<2>, bf.qr) % 16 == 0 && offsetof(BSmem<4>, bf.qr) % 16 == 0 &&
                  offsetof(BSmem<8>, bf.qr) % 16 == 0,
              "query pairs are read with 8-byte loads");

template <int G>
__global__ void __launch_bounds__(128, 4) bf16_kernel(BArgs a) {
  __shared__ BSmem<G> sm;
  pdl_trigger();
  part::bf16_role<G>(a, sm.bf, (int)blockIdx.x, sm.scratch, [&](int b, int kvh, part::BfSmem<G> &, bool &wait) {
    // q_rot of the segment's query heads (the demoted key's score): thread c sums column c of R_k
    wait = false;
    const PoolArgs &p = a.p;
    const int c = threadIdx.x;
    const float *R = p.R_k + (size_t)kvh * D * D + c;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;
    for (int i0 = 0; i0 < D; i0 += 16) {
      float rv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) rv[i] = R[(size_t)(i0 + i) * D];
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = fmaf(sm.bf.qr[i0 + i][h], rv[i], acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) sm.qrot[h][c] = acc[h];
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    return &sm.qrot[0][0];
  });
  // the merge waits for this grid: it must complete after the history kernel
  pdl_wait();
}

}  // namespace tc

// ---------------------------------------------------------------------------------------------
template <int G, int NG>
static int tc_resident() {
  static std::atomic<int> slots[kMaxDevices];
  return per_device(slots, [](int dev) {
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(tc::hist_kernel<G, NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::Cfg<G, NG>::SMEM);
    return sms;  // one history CTA per SM
  });
}

static int tc_sms(int G, int NG) {
#define OSCAR_TC_CASE(g, ng) \
  if (G == g && NG == ng) return tc_resident<g, ng>();
  OSCAR_TC_CASE(1, 1) OSCAR_TC_CASE(2, 1) OSCAR_TC_CASE(4, 1) OSCAR_TC_CASE(8, 1)
  OSCAR_TC_CASE(1, 2) OSCAR_TC_CASE(2, 2) OSCAR_TC_CASE(4, 2) OSCAR_TC_CASE(8, 2)
  OSCAR_TC_CASE(1, 4) OSCAR_TC_CASE(2, 4) OSCAR_TC_CASE(4, 4) OSCAR_TC_CASE(8, 4)
#undef OSCAR_TC_CASE
  return 148;
}

int tc_hist_ctas(const PoolArgs &p) {
  long long n = tc_sms(p.Hq / p.Hkv, p.ng);
  const long long cap = (long long)p.B * p.Hkv * p.max_pages;
  if (cap < n) n = cap;
  return (int)(n < 1 ? 1 : n);
}

static size_t tc_bq_bytes(int G, int NG) {
  const int ncol = 2 * G * NG, N = ncol <= 16 ? 16 : ((ncol + 15) / 16) * 16;
  return (size_t)N * 256 + ((G + G * NG) * 4 + 15) / 16 * 16;
}

// Workspace: [operand images, 16-byte aligned][partial slots]
size_t tc_ws_bytes(const PoolArgs &p) {
  const int G = p.Hq / p.Hkv;
  const size_t img = ((size_t)p.B * p.Hkv * tc_bq_bytes(G, p.ng) + 255) / 256 * 256;
  const size_t slots = (size_t)tc_hist_ctas(p) + (size_t)p.B * p.Hkv * 7;
  return img + slots * G * PART_STRIDE * sizeof(float);
}

template <int G, int NG>
static cudaError_t launch_tc_g(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                               cudaStream_t s, const uint16_t *k_new, const uint16_t *v_new) {
  using C = tc::Cfg<G, NG>;
  const float sm_log2 = sm_scale * 1.4426950408889634f;
  uint8_t *img = reinterpret_cast<uint8_t *>(ws);
  const size_t img_bytes = ((size_t)p.B * p.Hkv * C::BQ_BYTES + 255) / 256 * 256;
  float *part = reinterpret_cast<float *>(img + img_bytes);
  tc::HArgs h;
  h.p = p;
  h.bq = img;
  h.part = part;
  h.n_hist = tc_hist_ctas(p);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(tc::hist_kernel<G, NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM)) !=
      cudaSuccess)
    return e;
  if ((e = launch_pdl(tc::qrot_kernel<G, NG>, dim3(p.B * p.Hkv), dim3(256), 0, s, p, q, img, sm_log2)) != cudaSuccess)
    return e;
  profile_begin(OSCAR_PROFILE_HISTORY, s);
  if ((e = launch_pdl(tc::hist_kernel<G, NG>, dim3(h.n_hist), dim3(C::THREADS), C::SMEM, s, h)) != cudaSuccess)
    return e;
  profile_end(OSCAR_PROFILE_HISTORY, s);
  tc::BArgs b;
  b.p = p;
  b.q = q;
  b.sm_log2 = sm_log2;
  b.n_hist = h.n_hist;
  b.part = part;
  b.step = k_new != nullptr;
  b.k_new = k_new;
  b.v_new = v_new;
  if ((e = launch_pdl(tc::bf16_kernel<G>, dim3(p.B * p.Hkv * 5), dim3(128), 0, s, b)) != cudaSuccess) return e;
  return launch_merge_v1(p, part, h.n_hist, out, k_new, v_new, s);
}

template <int G>
static cudaError_t launch_tc_ng(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                                cudaStream_t s, const uint16_t *k_new, const uint16_t *v_new) {
  switch (p.ng) {
    case 1: return launch_tc_g<G, 1>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 2: return launch_tc_g<G, 2>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 4: return launch_tc_g<G, 4>(p, q, out, sm_scale, ws, s, k_new, v_new);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_tc(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                             cudaStream_t s, const uint16_t *k_new, const uint16_t *v_new) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_tc_ng<1>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 2: return launch_tc_ng<2>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 4: return launch_tc_ng<4>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 8: return launch_tc_ng<8>(p, q, out, sm_scale, ws, s, k_new, v_new);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oscar

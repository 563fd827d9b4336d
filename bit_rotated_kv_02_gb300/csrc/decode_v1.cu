// Decode attention over the three-segment pool, tensor-core version (group size 128).
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": the INT2 kernel
// unpacks the 2-bit codes, dequantizes with scale/zero point and accumulates in floating point; a
// BF16 kernel handles the sink and recent window; an online-softmax merge combines the results.
// "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract: a
// custom INT2 attention kernel compatible with paged KV-cache serving.
//
// Launches:
//   qrot_kernel   q_rot = q · R_k for every query head (row-vector convention), fp32, and per (sequence,
//                 KV head) the history consumers' query fragments (MMA B operands, score factors).
//   attn_kernel   BF16 CTAs (first block indices): 64 sink or recent tokens each, compensated FMA dot
//                 products, one partial per chunk.  History CTAs: the flattened (sequence, KV head, page) space is
//                 cut into equal contiguous ranges, one per CTA; a producer warp streams up to four
//                 pages of one segment per ring stage (codes and scale/zero rows) into shared memory
//                 with 1-D bulk async copies; four consumer warps each process one whole page per
//                 stage with warp MMAs (m16n8k16, f16 inputs, f32 accumulate) for Q.K and P.V, with a
//                 lazily rescaled online softmax; one (m, l, o_rot) partial per head is written per
//                 (CTA, segment).
//   merge_kernel  LSE-combines a segment's partials, un-rotates the history part (o · R_v^T),
//                 adds the BF16 part and normalises.
// The decode step (oscar_decode_step) uses the same three launches: the attention kernel reads only what
// the step leaves unchanged (the history before the step, the window slots other than the new token's,
// which it takes from k_new / v_new); two of its BF16 CTAs per (sequence, KV head), idle long before the
// history CTAs finish, perform the demotion (K in the sink CTA, V in the first window CTA) and write the
// demoted token as a partial of its own; the merge stores the new token and advances the pool counters.
//
// Exactness of the tensor-core arithmetic: a 2-bit code c placed in the low mantissa bits of an
// fp16 with a zero exponent field is the subnormal c * 4^k * 2^-24 (k = its bit position / 2), so
// codes enter the MMA exactly with one AND per two codes.  q_rot is split into two fp16 terms on a
// fixed-point grid (so that a token's code sums are exact), the softmax weights into two fp16 terms
// (hi + lo, 22 significant bits), both pre-scaled by powers of two (including 4^-k) so that fp16 holds
// them; scale and zero point are applied in fp32 outside the MMA:
//   score = scale * sum_c code_c q_c + zero * sum_c q_c,   o_rot = sum_t p_t scale_t code_t + sum_t p_t zero_t.
// Softmax values are kept in base 2 (scores pre-multiplied by log2 e), so partials carry log2 maxima.
#include "oscar_internal.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "bf16_part.cuh"
#include "split.cuh"

namespace oscar {

namespace v1 {

using part::StepState;
using part::step_state;
using split::npages_of;
using split::locate_range;

constexpr int NSTAGE = 3;
constexpr int PAGE_BYTES = 4608;   // Kc 2048 | Vc 2048 | Ks 128 | Kz 128 | Vs 128 | Vz 128
constexpr int CONSUMER_WARPS = 4, THREADS = 160;
constexpr int STAGE_PAGES = CONSUMER_WARPS;  // a stage holds up to one page of one segment per consumer warp
constexpr int STAGE_BYTES = PAGE_BYTES * STAGE_PAGES;
constexpr int OFF_KC = 0, OFF_VC = 2048, OFF_KS = 4096, OFF_KZ = 4224, OFF_VS = 4352, OFF_VZ = 4480;
constexpr int LAZY = 16;           // rescale the running output only when the max grows by > 2^16
constexpr int WEXP = 14 - LAZY;    // weights p * scale * 2^tau < 2^14 with tau = WEXP - e, scale < 2^e

struct Args {
  PoolArgs p;
  const float *qrot;   // [B][Hq][D] (qrot_kernel)
  const uint16_t *q;   // [B][Hq][D] bf16
  float sm_log2;       // softmax_scale * log2(e)
  int n_hist;          // history CTAs
  int n_bf;            // BF16 CTAs
  // block order: BF16 CTAs first (they and the history CTAs fit in one wave), or, when the BF16 CTAs
  // outnumber a sixth of the resident slots (large batches), the history CTAs first, so that they start at
  // once and the BF16 CTAs run in the remaining slots alongside them instead of in waves before them
  int hist_first;
  // dynamic tail of the history split (split::plan_of): enabled when the workspace holds its partial slots;
  // the chunk counter (zeroed by the query rotation) sits in the workspace after the partial slots
  int dyn;
  unsigned long long *dyn_ctr;
  float *part;         // partial slots [*][G][PART_STRIDE]
  const uint32_t *frag;  // per (sequence, KV head): the consumers' query fragments (qrot_kernel)
  // decode-step form: the pool counters still hold the state before the step (the merge kernel that
  // follows performs the demotion and the append); the BF16 CTAs attend the window after the step's
  // append and take the new token from k_new / v_new, the history CTAs the pages before the step.
  int step;
  const uint16_t *k_new, *v_new;  // [B][Hkv][D] bf16
};

// Unpack one 32-bit word of 16 codes (code j at bits 2j) into 8 fp16x2 registers at r[base..base+7]:
// register k holds (code k, code 8+k) as fp16 subnormals scaled by 4^k (k <= 4) or 4^(k-5) (k >= 5).
__device__ __forceinline__ void unpack16(uint32_t x, uint32_t (&r)[16], int base) {
#pragma unroll
  for (int k = 0; k < 5; ++k) r[base + k] = x & (0x00030003u << (2 * k));
  const uint32_t xs = x >> 10;
#pragma unroll
  for (int k = 0; k < 3; ++k) r[base + 5 + k] = xs & (0x00030003u << (2 * k));
}
// Indicator plane [c >= i] (i = 1, 2, 3) of the 2-bit fields of w, in each field's low bit: a code
// c = [c >= 1] + [c >= 2] + [c >= 3], and each plane unpacks like a code (an exact subnormal 0 or 4^k).
__device__ __forceinline__ uint32_t plane_ge(uint32_t w, int i) {
  return i == 1 ? (w | (w >> 1)) & 0x55555555u : i == 2 ? (w >> 1) & 0x55555555u : (w & (w >> 1)) & 0x55555555u;
}
__device__ __forceinline__ float code_factor_inv(int k) {  // 1 / 4^k' for register k (0..7)
  const int e = (k <= 4) ? 2 * k : 2 * (k - 5);
  return __int_as_float((127 - e) << 23);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }

template <int G>
struct Smem {
  static constexpr int NT = (2 * G + 7) / 8;
  alignas(128) uint8_t ring[NSTAGE][STAGE_BYTES];
  uint64_t full[NSTAGE][STAGE_PAGES], empty[NSTAGE][STAGE_PAGES];  // one pair per page slot
  uint64_t csync;                                                    // consumer-warp barrier
  int meta_seg[NSTAGE], meta_ntok[NSTAGE][STAGE_PAGES], meta_flags[NSTAGE];  // flags: 1 last, 2 abort
  int meta_slot[NSTAGE];                                                      // partial slot of the stage
  alignas(16) float qr[D][G];  // BF16 CTAs: the queries, channel-major (read in 8-byte pairs)
  float wm[CONSUMER_WARPS][G], wl[CONSUMER_WARPS][G], wz[CONSUMER_WARPS][G];
  float wo[CONSUMER_WARPS][G][D];
  float pbuf[CONSUMER_WARPS][G][16];
  long long range_lo, range_n, n_dyn;
  int b0, kvh0, local0, np0, hl0;
};
static_assert(offsetof(Smem<2>, qr) % 16 == 0 && offsetof(Smem<4>, qr) % 16 == 0 && offsetof(Smem<8>, qr) % 16 == 0,
              "query pairs are read with 8-byte loads");

// Query fragments of one (sequence, KV head) as the history consumers use them: per MMA lane, the B
// operands bq[nt][j][hb] (NT * 16 words) and the score factors kf[nt], zf[nt] of the lane's accumulator
// columns, stored word-major ([word][32 lanes]) so that a warp loads each word coalesced.
template <int G>
__host__ __device__ constexpr int frag_words() { return Smem<G>::NT * 18; }

// ---------------------------------------------------------------------------------------------
// q_rot = q . R_k for the G query heads of one (sequence, KV head) and the history consumers' query
// fragments (frag_words per lane): grid B * Hkv, 512 threads.  Thread (c, quarter) sums rows 16k ..
// 16k+15 for k = 2 quarter, 2 quarter + 1 of column c; the eight partial sums are added pairwise.  Per
// head the exponent sigma with amax(q_rot) * 2^sigma < 2^14, kf = 2^(24 - sigma) * log2(e) *
// softmax_scale and zf = sum(q_rot) * log2(e) * softmax_scale, and per lane the q_rot values of its B
// operands: y = q_rot * 2^sigma split on a fixed-point grid, hi = 8 rint(y / 8) and lo = rint((y - hi) *
// 256) / 256 (so |y - hi - lo| <= 2^-9 < 2^-23 amax(y)), each scaled by 4^-k for the code placed at bit
// 2k of its 16-bit lane.  Every product of a code with hi is an integer multiple of 2^-21 and every
// product with lo a multiple of 2^-32, and 128 of them stay below 2^24 units: the tensor cores' float32
// sums of a token's code products are exact, whatever their order.
// The loads of q and R_k (inputs no kernel of the step writes) are issued before the griddepcontrol.wait;
// the trigger follows the wait, so that the attention kernel, which reads the pool counters at once,
// starts only after the previous step's merge has completed.
template <int G>
__global__ void __launch_bounds__(512) qrot_kernel(PoolArgs p, const uint16_t *q, float *qrot, uint32_t *frag,
                                                   float sm_log2, unsigned long long *dyn_ctr) {
  constexpr int NT = Smem<G>::NT;
  __shared__ float qs[G][D];
  __shared__ float part[8][G][D];
  __shared__ int s_sig[8];
  __shared__ float s_kf[8], s_zf[8];
  const int s = blockIdx.x, b = s / p.Hkv, kvh = s % p.Hkv;
  const int tid = threadIdx.x, c = tid & (D - 1), qt = tid >> 7;
  const float *R = p.R_k + (size_t)kvh * D * D + (size_t)(32 * qt) * D + c;
  float r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = R[(size_t)i * D];
  constexpr int QPT = (G * D + 511) / 512;
  uint16_t qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int i = tid + 512 * k;
    qv[k] = i < G * D ? q[((size_t)b * p.Hq + kvh * G) * D + i] : 0;
  }
  pdl_wait();  // the previous kernel on the stream (the last reader of q_rot and the fragments) has completed
  pdl_trigger();
  if (dyn_ctr != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *dyn_ctr = 0;  // the split's chunk counter
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int i = tid + 512 * k;
    if (i < G * D) qs[i / D][i % D] = bf16_to_f32(qv[k]);
  }
  __syncthreads();
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc = fmaf(qs[h][32 * qt + 16 * hf + i], r[16 * hf + i], acc);
      part[2 * qt + hf][h][c] = acc;
    }
  }
  __syncthreads();
  if (qt == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float v = ((part[0][h][c] + part[1][h][c]) + (part[2][h][c] + part[3][h][c])) +
                      ((part[4][h][c] + part[5][h][c]) + (part[6][h][c] + part[7][h][c]));
      qrot[((size_t)b * p.Hq + kvh * G + h) * D + c] = v;
      qs[h][c] = v;  // q is no longer needed
    }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < G) {
    const int h = warp;
    float amax = 0.f, sum = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float v = qs[h][lane + 32 * k];
      amax = fmaxf(amax, fabsf(v));
      sum += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, o));
      sum += __shfl_xor_sync(FULL, sum, o);
    }
    if (lane == 0) {
      int e = 0;
      if (amax > 0.f) frexpf(amax, &e);
      const int sig = (amax > 0.f) ? 14 - e : 0;  // amax * 2^sig < 2^14
      s_sig[h] = sig;
      s_kf[h] = pow2f(24 - sig) * sm_log2;
      s_zf[h] = sum * sm_log2;
    }
  }
  __syncthreads();
  if (warp < NT) {
    const int nt = warp, gq = lane >> 2, t = lane & 3;
    uint32_t *fr = frag + (size_t)s * frag_words<G>() * 32 + lane;
    const int h = 4 * nt + (gq >> 1), split = gq & 1;
    const bool live = h < G;
    const float s2 = live ? pow2f(s_sig[h]) : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int i = 2 * j + hb;  // register index of the token's 16 (word i/8, slot i%8)
        const int wi = i >> 3, k = i & 7;
        const int ch_lo = 32 * t + 16 * wi + k, ch_hi = ch_lo + 8;
        const float f = code_factor_inv(k);
        float v[2];
        const int chs[2] = {ch_lo, ch_hi};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float y = live ? qs[min(h, G - 1)][chs[e]] * s2 : 0.f;  // exact: s2 is a power of two
          const float hi = 8.f * rintf(y * 0.125f);
          const float lo = rintf((y - hi) * 256.f) * (1.f / 256.f);
          v[e] = (split == 0 ? hi : lo) * f;
        }
        fr[(nt * 16 + i) * 32] = pack_half2(v[0], v[1]);
      }
    }
    const int hc = min(4 * nt + t, G - 1);  // accumulator column pair (2t, 2t+1) = head 4 nt + t
    fr[(NT * 16 + nt) * 32] = __float_as_uint(s_kf[hc]);
    fr[(NT * 16 + NT + nt) * 32] = __float_as_uint(s_zf[hc]);
  }
}

// ---------------------------------------------------------------------------------------------
template <int G>
struct WarpState {
  static constexpr int NT = (2 * G + 7) / 8;
  float m2[NT], l[NT], oz[NT];
  float O[NT][8][4];
  int tau;        // weight scaling exponent (o accumulates in units of 2^-24 * 2^-tau per code step)
  float tau_lim;  // largest V scale the current tau admits (0 until the first non-zero scale)
  uint32_t csync_par;  // phase parity of the consumer barrier
};

// Barrier among the consumer warps: an mbarrier counting one arrival per warp, waited with a time
// limit, so that no thread can wait forever when a warp has left the pipeline after a timeout (the
// error bit is set and the results of the launch are not valid).
template <int G>
__device__ __forceinline__ void consumer_sync(Smem<G> &sm, uint32_t &par, uint32_t *err) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.csync);
  const bool ok = __all_sync(FULL, mbar_wait_bounded(&sm.csync, par));
  par ^= 1u;
  if (!ok && (threadIdx.x & 31) == 0) atomicOr(err, OSCAR_DEVERR_TIMEOUT);
}

template <int G>
__device__ __forceinline__ void reset(WarpState<G> &ws) {
#pragma unroll
  for (int nt = 0; nt < WarpState<G>::NT; ++nt) {
    ws.m2[nt] = -INFINITY; ws.l[nt] = 0.f; ws.oz[nt] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) ws.O[nt][mt][r] = 0.f;
  }
  ws.tau = 0;
  ws.tau_lim = 0.f;
}

// Segment setup (consumer threads only): load q_rot, derive per-head scaling, build B fragments.
// Codebook levels of one KV head as the history consumers use them: l[c] = l0 + sum_{i < c} d[i]
// (pools without a codebook for K or V use 0, 1, 2, 3); dvmax = max d[i] of V bounds the weight range.
struct Levels {
  float l0k, dk[3], l0v, dv[3], dvmax;
};

template <int G, bool CB>
__device__ __forceinline__ void setup_segment(const Args &a, int b, int kvh, uint32_t (&bq)[Smem<G>::NT][8][2],
                                              float (&kf)[Smem<G>::NT], float (&zf)[Smem<G>::NT], Levels &lv) {
  constexpr int NT = Smem<G>::NT;
  if (CB) {
    const float4 ck = a.p.cb_k != nullptr ? reinterpret_cast<const float4 *>(a.p.cb_k)[kvh] : make_float4(0.f, 1.f, 2.f, 3.f);
    const float4 cv = a.p.cb_v != nullptr ? reinterpret_cast<const float4 *>(a.p.cb_v)[kvh] : make_float4(0.f, 1.f, 2.f, 3.f);
    lv.l0k = ck.x; lv.dk[0] = ck.y - ck.x; lv.dk[1] = ck.z - ck.y; lv.dk[2] = ck.w - ck.z;
    lv.l0v = cv.x; lv.dv[0] = cv.y - cv.x; lv.dv[1] = cv.z - cv.y; lv.dv[2] = cv.w - cv.z;
    lv.dvmax = fmaxf(fmaxf(lv.dv[0], lv.dv[1]), lv.dv[2]);
  }
  if (a.step) pdl_wait();  // the step's query rotation (the previous kernel on this stream) has completed
  const uint32_t *fr = a.frag + (size_t)(b * a.p.Hkv + kvh) * frag_words<G>() * 32 + (threadIdx.x & 31);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int i = 0; i < 16; ++i) bq[nt][i >> 1][i & 1] = fr[(nt * 16 + i) * 32];
    kf[nt] = __uint_as_float(fr[(NT * 16 + nt) * 32]);
    zf[nt] = __uint_as_float(fr[(NT * 16 + NT + nt) * 32]);
  }
}

// Flush the consumer warps' state for one segment into partial slot `slot`.
template <int G>
__device__ __forceinline__ void flush(const Args &a, Smem<G> &sm, WarpState<G> &ws, float *slot) {
  constexpr int NT = Smem<G>::NT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float l = ws.l[nt], oz = ws.oz[nt];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l += __shfl_xor_sync(FULL, l, o);
      oz += __shfl_xor_sync(FULL, oz, o);
    }
    const int h = 4 * nt + t;
    if (h < G) {
      if (gq == 0) { sm.wm[warp][h] = ws.m2[nt]; sm.wl[warp][h] = l; sm.wz[warp][h] = oz; }
      const float unit = pow2f(24 - ws.tau);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int i = 2 * mt + r;
          const int ch = 16 * gq + i;
          sm.wo[warp][h][ch] = (ws.O[nt][mt][2 * r] + ws.O[nt][mt][2 * r + 1]) * unit * code_factor_inv(i & 7);
        }
    }
  }
  consumer_sync(sm, ws.csync_par, a.p.err);
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < CONSUMER_WARPS; ++w) M = fmaxf(M, sm.wm[w][h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < CONSUMER_WARPS; ++w) {
        const float e = sm.wm[w][h] == -INFINITY ? 0.f : exp2f(sm.wm[w][h] - M);
        L += e * sm.wl[w][h];
        O += e * (sm.wo[w][h][tid] + sm.wz[w][h]);
      }
    }
    slot[h * PART_STRIDE + tid] = O;
    if (tid == 0) { slot[h * PART_STRIDE + D] = M; slot[h * PART_STRIDE + D + 1] = L; }
  }
  consumer_sync(sm, ws.csync_par, a.p.err);
  reset(ws);
}

// 8x8 transpose of a matrix of 16-bit values held one 32-bit pair per lane in the mma fragment
// layout (lane (g, t) holds row g, columns 2t and 2t+1); the result is in the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

// One page in one consumer warp: all 64 tokens as four 16-row MMA tiles; ntok = valid tokens (1..64).
// MMA row 16 mt + g (+ 8) of tile mt holds token 8 g + 2 mt (+ 1), so lane (g, t) owns the eight
// consecutive tokens 8 g .. 8 g + 7 (its accumulator rows j = 2 mt + e) and reads their scale/zero
// rows with one 16-byte load per array.  The softmax weights are formed in the QK accumulator layout
// (column pair 2t, 2t+1 = head t's hi and lo query terms), split into fp16 hi + lo and transposed with
// movmatrix into the B operand of the P.V products, whose A operand therefore takes, for k-index
// pairs (2t, 2t+1) and (2t+8, 2t+9) of tile mt, the tokens 16 t + 2 mt (+ 8) and 16 t + 2 mt + 1 (+ 8).
// Rows past ntok are masked: score -inf, value scale and zero 0 (their codes are finite integers).
// CB: codebook levels.  Q.K takes the three indicator planes [c >= i] through the same query fragments
// (their sums stay exact) and combines them as l0 * sum(q) + sum_i d_k[i] * plane_i; P.V takes the planes
// against the weights scaled by d_v[i]; the zero points absorb scale * l0.
template <int G, bool CB>
__device__ __forceinline__ void page_pass(const uint8_t *pb, int ntok, WarpState<G> &ws,
                                          const uint32_t (&bq)[Smem<G>::NT][8][2], const float (&kf_)[Smem<G>::NT],
                                          const float (&zf_)[Smem<G>::NT], const Levels &lv) {
  constexpr int NT = Smem<G>::NT;
  constexpr bool ALL_LIVE = (G % 4) == 0;
  const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
  // ---- QK: A = K codes (lane t owns channels 32t .. 32t+31 of its two tokens per tile) ----
  float S[4][NT][4];
  const uint8_t *kc = pb + OFF_KC + gq * 256 + 8 * t;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) S[mt][nt][0] = S[mt][nt][1] = S[mt][nt][2] = S[mt][nt][3] = 0.f;
    const uint2 ka = *reinterpret_cast<const uint2 *>(kc + 64 * mt);
    const uint2 kb = *reinterpret_cast<const uint2 *>(kc + 64 * mt + 32);
    if (!CB) {
      uint32_t T0[16], T1[16];
      unpack16(ka.x, T0, 0); unpack16(ka.y, T0, 8);
      unpack16(kb.x, T1, 0); unpack16(kb.y, T1, 8);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mma16816(S[mt][nt], T0[2 * j], T1[2 * j], T0[2 * j + 1], T1[2 * j + 1], bq[nt][j][0], bq[nt][j][1]);
    } else {
      float T[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) T[nt][0] = T[nt][1] = 0.f;
#pragma unroll
      for (int i = 1; i <= 3; ++i) {
        float Si[NT][4];
        uint32_t T0[16], T1[16];
        unpack16(plane_ge(ka.x, i), T0, 0); unpack16(plane_ge(ka.y, i), T0, 8);
        unpack16(plane_ge(kb.x, i), T1, 0); unpack16(plane_ge(kb.y, i), T1, 8);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          Si[nt][0] = Si[nt][1] = Si[nt][2] = Si[nt][3] = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            mma16816(Si[nt], T0[2 * j], T1[2 * j], T0[2 * j + 1], T1[2 * j + 1], bq[nt][j][0], bq[nt][j][1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) T[nt][e] = fmaf(lv.dk[i - 1], Si[nt][2 * e] + Si[nt][2 * e + 1], T[nt][e]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        S[mt][nt][0] = T[nt][0]; S[mt][nt][1] = 0.f;
        S[mt][nt][2] = T[nt][1]; S[mt][nt][3] = 0.f;
      }
    }
  }
  // ---- scale / zero of the lane's tokens 8g .. 8g+7 ----
  const uint4 ks4 = *reinterpret_cast<const uint4 *>(pb + OFF_KS + 16 * gq);
  const uint4 kz4 = *reinterpret_cast<const uint4 *>(pb + OFF_KZ + 16 * gq);
  const uint4 vs4 = *reinterpret_cast<const uint4 *>(pb + OFF_VS + 16 * gq);
  const uint4 vz4 = *reinterpret_cast<const uint4 *>(pb + OFF_VZ + 16 * gq);
  const int nvalid = ntok - 8 * gq;  // rows j < nvalid are tokens of the page
  float ks[8], kz[8], vs[8], vz[8];
  {
    const uint32_t kw[4] = {ks4.x, ks4.y, ks4.z, ks4.w}, zw[4] = {kz4.x, kz4.y, kz4.z, kz4.w};
    const uint32_t vw[4] = {vs4.x, vs4.y, vs4.z, vs4.w}, uw[4] = {vz4.x, vz4.y, vz4.z, vz4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ks[2 * i] = __uint_as_float(kw[i] << 16); ks[2 * i + 1] = __uint_as_float(kw[i] & 0xffff0000u);
      kz[2 * i] = __uint_as_float(zw[i] << 16); kz[2 * i + 1] = __uint_as_float(zw[i] & 0xffff0000u);
      vs[2 * i] = __uint_as_float(vw[i] << 16); vs[2 * i + 1] = __uint_as_float(vw[i] & 0xffff0000u);
      vz[2 * i] = __uint_as_float(uw[i] << 16); vz[2 * i + 1] = __uint_as_float(uw[i] & 0xffff0000u);
    }
  }
  if (CB) {  // zero points that absorb scale * l0
#pragma unroll
    for (int j = 0; j < 8; ++j) { kz[j] = fmaf(ks[j], lv.l0k, kz[j]); vz[j] = fmaf(vs[j], lv.l0v, vz[j]); }
  }
  if (nvalid < 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j >= nvalid) { vs[j] = 0.f; vz[j] = 0.f; }
  }
  // ---- weight scaling exponent tau: weights p * vs * 2^tau stay below 2^14 ----
  // (a warp vote on the lane maxima; the cross-lane maximum is formed only when tau must change)
  float vmax = fmaxf(max3f(vs[0], vs[1], vs[2]), max3f(max3f(vs[3], vs[4], vs[5]), vs[6], vs[7]));
  if (CB) vmax *= lv.dvmax;  // the largest weight factor of the three planes
  if (__any_sync(FULL, vmax >= ws.tau_lim && vmax > 0.f)) {
    vmax = fmaxf(vmax, __shfl_xor_sync(FULL, vmax, 4));
    vmax = fmaxf(vmax, __shfl_xor_sync(FULL, vmax, 8));
    vmax = fmaxf(vmax, __shfl_xor_sync(FULL, vmax, 16));
    int e;
    frexpf(vmax, &e);
    const int tnew = max(-100, min(100, WEXP - e));
    if (ws.tau_lim > 0.f && tnew < ws.tau) {
      const float f = pow2f(tnew - ws.tau);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int m8 = 0; m8 < 8; ++m8)
#pragma unroll
          for (int r = 0; r < 4; ++r) ws.O[nt][m8][r] *= f;
    }
    if (ws.tau_lim == 0.f || tnew < ws.tau) ws.tau = tnew;
    ws.tau_lim = pow2f(WEXP - ws.tau);
  }
  const float untau = pow2f(-ws.tau);
  // ---- scores, lazily rescaled online softmax, weights ----
  uint32_t bw[CB ? 3 : 1][NT][4][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = ALL_LIVE ? 4 * nt + t : min(4 * nt + t, G - 1);
    const bool live_h = ALL_LIVE || 4 * nt + t < G;
    const float kf = kf_[nt], zf = zf_[nt];
    (void)h;
    // score of row j = 2 mt + e: (S hi + S lo) * ks * kf + kz * zf, both rows of a tile in one paired op
    float sc[8];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const float2 x = make_float2(S[mt][nt][0] + S[mt][nt][1], S[mt][nt][2] + S[mt][nt][3]);
      const float2 v = ffma2(fmul2(x, make_float2(ks[2 * mt], ks[2 * mt + 1])), make_float2(kf, kf),
                             fmul2(make_float2(kz[2 * mt], kz[2 * mt + 1]), make_float2(zf, zf)));
      sc[2 * mt] = v.x;
      sc[2 * mt + 1] = v.y;
    }
    if (nvalid < 8) {  // a partial page: rows past its last token
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j >= nvalid) sc[j] = -INFINITY;
    }
    // lazy rescaling: the head's maximum is formed across lanes only when some row exceeds the
    // reference by more than 2^LAZY (a warp vote on the lane maxima decides)
    float tmax = fmaxf(max3f(sc[0], sc[1], sc[2]), max3f(max3f(sc[3], sc[4], sc[5]), sc[6], sc[7]));
    if (__any_sync(FULL, tmax > ws.m2[nt] + (float)LAZY)) {
      tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, 16));
      if (tmax > ws.m2[nt] + (float)LAZY) {
        const float alpha = (ws.m2[nt] == -INFINITY) ? 0.f : fast_exp2(ws.m2[nt] - tmax);
        ws.l[nt] *= alpha;
        ws.oz[nt] *= alpha;
#pragma unroll
        for (int m8 = 0; m8 < 8; ++m8)
#pragma unroll
          for (int r = 0; r < 4; ++r) ws.O[nt][m8][r] *= alpha;
        ws.m2[nt] = tmax;
      }
    }
    // p * 2^tau = exp2(score - (m - tau)); l and the zero-point sum take p itself
    const float mref = ws.m2[nt] - (float)ws.tau;
    float2 lsum = make_float2(0.f, 0.f), zsum = make_float2(0.f, 0.f);
    float wv[8];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const float2 d = fsub2(make_float2(sc[2 * mt], sc[2 * mt + 1]), make_float2(mref, mref));
      const float2 pr = make_float2(fast_exp2(d.x), fast_exp2(d.y));  // 0 for rows past ntok (score -inf)
      lsum = fadd2(lsum, pr);
      zsum = ffma2(pr, make_float2(vz[2 * mt], vz[2 * mt + 1]), zsum);
      const float2 w = fmul2(pr, make_float2(vs[2 * mt], vs[2 * mt + 1]));
      wv[2 * mt] = live_h ? w.x : 0.f;
      wv[2 * mt + 1] = live_h ? w.y : 0.f;
    }
    ws.l[nt] = fmaf(lsum.x + lsum.y, untau, ws.l[nt]);
    ws.oz[nt] = fmaf(zsum.x + zsum.y, untau, ws.oz[nt]);
#pragma unroll
    for (int pl = 0; pl < (CB ? 3 : 1); ++pl) {
      uint32_t wp[8];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        float2 w = make_float2(wv[2 * mt], wv[2 * mt + 1]);
        if (CB) w = fmul2(w, make_float2(lv.dv[pl], lv.dv[pl]));
        const float2 hi = make_float2(__uint_as_float(__float_as_uint(w.x) & 0xffffe000u),   // w to 11
                                      __uint_as_float(__float_as_uint(w.y) & 0xffffe000u));  // significant bits
        const float2 lo = fsub2(w, hi);
        wp[2 * mt] = pack_half2(hi.x, lo.x);  // (hi, lo)
        wp[2 * mt + 1] = pack_half2(hi.y, lo.y);
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        bw[pl][nt][mt][0] = movmatrix_trans(wp[2 * mt]);
        bw[pl][nt][mt][1] = movmatrix_trans(wp[2 * mt + 1]);
      }
    }
  }
  // ---- P.V per tile: A = V codes^T (group g: channels 16g .. 16g+15, one 32-bit word per token) ----
  const uint32_t *vrow = reinterpret_cast<const uint32_t *>(pb + OFF_VC) + 16 * t * 8 + gq;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    const uint32_t xa = vrow[16 * mt], xb = vrow[64 + 16 * mt];           // tokens 16t+2mt, 16t+8+2mt
    const uint32_t xc = vrow[16 * mt + 8], xd = vrow[64 + 16 * mt + 8];   // the same + 1
    const uint32_t w0 = prmt(xa, xb, 0x5410), w1 = prmt(xa, xb, 0x7632);
    const uint32_t w2 = prmt(xc, xd, 0x5410), w3 = prmt(xc, xd, 0x7632);
#pragma unroll
    for (int pl = 0; pl < (CB ? 3 : 1); ++pl) {
      uint32_t VA[16], VB[16];
      if (CB) {
        unpack16(plane_ge(w0, pl + 1), VA, 0); unpack16(plane_ge(w1, pl + 1), VA, 8);
        unpack16(plane_ge(w2, pl + 1), VB, 0); unpack16(plane_ge(w3, pl + 1), VB, 8);
      } else {
        unpack16(w0, VA, 0); unpack16(w1, VA, 8);
        unpack16(w2, VB, 0); unpack16(w3, VB, 8);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int m8 = 0; m8 < 8; ++m8)
          mma16816(ws.O[nt][m8], VA[2 * m8], VA[2 * m8 + 1], VB[2 * m8], VB[2 * m8 + 1], bw[pl][nt][mt][0],
                   bw[pl][nt][mt][1]);
    }
  }
}

// DYN: the build of the kernel with the dynamic tail of the split (launched when the pool can be large enough
// for it); without it the producer issues its static range only and the consumers flush on segment changes.
template <int G, bool CB, bool DYN>
__device__ __forceinline__ void hist_role(const Args &a, Smem<G> &sm, const int cta) {
  constexpr int NT = Smem<G>::NT;
  const PoolArgs &p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s)
      for (int pg = 0; pg < STAGE_PAGES; ++pg) { mbar_init(&sm.full[s][pg], 1); mbar_init(&sm.empty[s][pg], 1); }
    mbar_init(&sm.csync, CONSUMER_WARPS);
    mbar_fence_init();
  }
  split::Plan pl{};
  if (warp == CONSUMER_WARPS) {  // the producer warp locates this CTA's range
    long long lo, n;
    int b0, kvh0, local0, np0, hl0;
    locate_range(p, a.n_hist, cta, DYN, lo, n, b0, kvh0, local0, np0, hl0, pl);
    if (lane == 0) {
      sm.range_lo = lo; sm.range_n = n; sm.b0 = b0; sm.kvh0 = kvh0; sm.local0 = local0; sm.np0 = np0; sm.hl0 = hl0;
      sm.n_dyn = pl.n_dyn;
    }
  }
  __syncthreads();
  const long long n = sm.range_n;
  if (n <= 0 && (!DYN || sm.n_dyn == 0)) return;

  if (warp == CONSUMER_WARPS) {
    // ---------------- producer warp: up to STAGE_PAGES pages of one segment per stage ----------------
    // Lane i owns page i of a stage and issues its bulk copies.  The page-table entries are read 32 at a
    // time (lane i holds entry pt_base + i of sequence b; every KV head of a sequence shares them), so
    // that most stages issue their copies without a round trip of their own.  hist_len is read once per
    // sequence.  A stage carries its partial slot (slot0 + segment: the static range's slot0 = cta, chunk
    // k's dyn_slot0 + k); the consumers flush when it changes.
    const uint64_t stream_pol = l2_evict_first();
    int stage = 0, it = 0;
    uint32_t phase = 0;
    int pt_base = -1, pt_b = -1, ptv = -1;
    int last_seg = sm.b0 * p.Hkv + sm.kvh0, last_slot = -1;
    bool abort = false;
    // pages [start, start + cnt_all) from position (b, kvh, local); `final` marks the stage that ends the CTA
    auto issue = [&](long long cnt_all, int b, int kvh, int local, int np, int hl, int slot0, bool final) {
      long long done = 0;
      while (done < cnt_all && !abort) {
        if (it >= NSTAGE) {  // every page slot of the stage released by its consumer warp
          bool okw = true;
          if (lane < STAGE_PAGES) okw = mbar_wait_bounded(&sm.empty[stage][lane], phase ^ 1);
          abort = !__all_sync(FULL, okw);
          if (abort && lane == 0) atomicOr(p.err, OSCAR_DEVERR_TIMEOUT);
        }
        const int seg = b * p.Hkv + kvh;
        const int cnt = abort ? 0 : (int)min((long long)STAGE_PAGES, min(cnt_all - done, (long long)(np - local)));
        if (cnt <= 0 && !abort) {  // counters inconsistent with the range (changed during the launch): stop
          abort = true;
          if (lane == 0) atomicOr(p.err, OSCAR_DEVERR_COUNTERS);
        }
        if (cnt > 0 && (b != pt_b || local < pt_base || local + cnt > pt_base + 32)) {
          pt_b = b;
          pt_base = local;
          ptv = local + lane < np ? ld_hint(p.page_table + (size_t)b * p.max_pages + local + lane, l2_evict_last()) : -1;
        }
        int pp = __shfl_sync(FULL, ptv, (local - pt_base + lane) & 31), ntk = 0;
        if (lane >= cnt) pp = -1;
        if (lane < cnt) {
          const int lp = local + lane;
          ntk = min(PAGE, hl - lp * PAGE);
          if (pp < 0 || pp >= p.num_pages) {
            atomicOr(p.err, OSCAR_DEVERR_PAGE_INDEX);
            pp = -1;
          }
        }
        const bool have = pp >= 0;
        if (lane < STAGE_PAGES) sm.meta_ntok[stage][lane] = have ? ntk : 0;
        if (lane == 0) {
          sm.meta_seg[stage] = seg;
          if constexpr (DYN) sm.meta_slot[stage] = slot0 + seg;
          sm.meta_flags[stage] = ((final && done + cnt >= cnt_all) ? 1 : 0) | (abort ? 2 : 0);
        }
        if constexpr (DYN) {
          last_seg = seg;
          last_slot = slot0 + seg;
        }
        __syncwarp();  // the stage's metadata is written before any of its slots can complete
        if (lane < STAGE_PAGES) {
          uint64_t *bar = &sm.full[stage][lane];
          if (have) {
            mbar_arrive_expect_tx(bar, (uint32_t)PAGE_BYTES);
            uint8_t *dst = sm.ring[stage] + lane * PAGE_BYTES;
            const size_t row = ((size_t)pp * p.Hkv + kvh) * PAGE;
            bulk_g2s_hint(dst + OFF_KC, p.codes_k + row * (D / 4), 2048, bar, stream_pol);
            bulk_g2s_hint(dst + OFF_VC, p.codes_v + row * (D / 4), 2048, bar, stream_pol);
            bulk_g2s_hint(dst + OFF_KS, p.scale_k + row, 128, bar, stream_pol);
            bulk_g2s_hint(dst + OFF_KZ, p.zero_k + row, 128, bar, stream_pol);
            bulk_g2s_hint(dst + OFF_VS, p.scale_v + row, 128, bar, stream_pol);
            bulk_g2s_hint(dst + OFF_VZ, p.zero_v + row, 128, bar, stream_pol);
          } else {
            mbar_arrive(bar);
          }
        }
        if (abort) {
          // wait (bounded) for the copies still in flight into stages the consumers may not read
          if (lane < STAGE_PAGES)
            for (int k = max(0, it - NSTAGE + 1); k < it; ++k)
              mbar_wait_bounded(&sm.full[k % NSTAGE][lane], (uint32_t)((k / NSTAGE) & 1));
          return;
        }
        done += cnt;
        local += cnt;
        if (local == np && done < cnt_all) {
          local = 0;
          if (++kvh == p.Hkv) {
            kvh = 0;
            do { ++b; } while (b < p.B && npages_of(p, b) == 0);
            if (b < p.B) {
              np = npages_of(p, b);
              hl = max(0, min(split::hist_len_of(p, b), p.max_pages * PAGE));
            }
          }
        }
        ++it;
        if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
      }
    };
    // the static range, then (dynamic tail) chunks while any are left; one call site of issue() keeps the
    // producer's code small
    const bool dyn = DYN && sm.n_dyn > 0;
    const long long dyn_slot0 = (long long)a.n_hist + 7LL * p.B * p.Hkv;
    bool static_done = n <= 0, waited = false;
    while (!abort) {
      long long cnt_all;
      int b, kvh, local, np, hl, slot0;
      bool final;
      if (!static_done) {
        static_done = true;
        cnt_all = n; b = sm.b0; kvh = sm.kvh0; local = sm.local0; np = sm.np0; hl = sm.hl0; slot0 = cta;
        final = !dyn;
      } else {
        if (!dyn) break;
        if (!waited) {  // the chunk counter was zeroed by the query rotation, complete after this wait
          pdl_wait();
          waited = true;
        }
        long long k = 0;
        if (lane == 0) k = (long long)atomicAdd(a.dyn_ctr, 1ull);
        k = __shfl_sync(FULL, k, 0);
        if (k >= pl.n_dyn) break;
        const long long start = pl.static_pages + k * pl.dyn_pages;
        cnt_all = min(pl.dyn_pages, pl.total - start);
        split::locate_at(p, start, b, kvh, local, np, hl);
        slot0 = (int)(dyn_slot0 + k);
        final = false;
      }
      issue(cnt_all, b, kvh, local, np, hl, slot0, final);
    }
    if (DYN && dyn) {
      if (!abort) {
        // the terminal stage: no pages, the last slot (no flush), the end flag
        if (it >= NSTAGE) {
          bool okw = true;
          if (lane < STAGE_PAGES) okw = mbar_wait_bounded(&sm.empty[stage][lane], phase ^ 1);
          abort = !__all_sync(FULL, okw);
          if (abort && lane == 0) atomicOr(p.err, OSCAR_DEVERR_TIMEOUT);
        }
        if (lane < STAGE_PAGES) sm.meta_ntok[stage][lane] = 0;
        if (lane == 0) {
          sm.meta_seg[stage] = last_seg;
          sm.meta_slot[stage] = last_slot;
          sm.meta_flags[stage] = 1 | (abort ? 2 : 0);
        }
        __syncwarp();
        if (lane < STAGE_PAGES) mbar_arrive(&sm.full[stage][lane]);
      }
    }
    return;
  }
  // ---------------- consumers ----------------
  WarpState<G> ws;
  reset(ws);
  uint32_t bq[NT][8][2];
  float kf[NT], zf[NT];
  // the first segment's query setup needs no pages: it overlaps the first bulk copies
  int cur = sm.b0 * p.Hkv + sm.kvh0, cur_slot = -1, stage = 0;
  ws.csync_par = 0;
  Levels lv{};
  setup_segment<G, CB>(a, sm.b0, sm.kvh0, bq, kf, zf, lv);
  uint32_t phase = 0;
  while (true) {
    if (!mbar_wait_bounded(&sm.full[stage][warp], phase)) {
      if (lane == 0) atomicOr(a.p.err, OSCAR_DEVERR_TIMEOUT);
      break;
    }
    const int flags = sm.meta_flags[stage];
    if (flags & 2) break;  // producer aborted
    const int seg = sm.meta_seg[stage];
    if constexpr (DYN) {
      const int slot = sm.meta_slot[stage];
      if (slot != cur_slot) {
        if (cur_slot >= 0) flush(a, sm, ws, a.part + (size_t)cur_slot * G * PART_STRIDE);
        cur_slot = slot;
        if (seg != cur) {
          cur = seg;
          setup_segment<G, CB>(a, seg / p.Hkv, seg % p.Hkv, bq, kf, zf, lv);
        }
      }
    } else if (seg != cur) {
      flush(a, sm, ws, a.part + ((size_t)cta + cur) * G * PART_STRIDE);
      cur = seg;
      setup_segment<G, CB>(a, seg / p.Hkv, seg % p.Hkv, bq, kf, zf, lv);
    }
    const int ntok = sm.meta_ntok[stage][warp];
    const uint8_t *pb = sm.ring[stage] + warp * PAGE_BYTES;
    if (ntok > 0) page_pass<G, CB>(pb, ntok, ws, bq, kf, zf, lv);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage][warp]);
    if (flags & 1) break;
    if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
  }
  if constexpr (DYN) {
    if (cur_slot >= 0) flush(a, sm, ws, a.part + (size_t)cur_slot * G * PART_STRIDE);
  } else {
    flush(a, sm, ws, a.part + ((size_t)cta + cur) * G * PART_STRIDE);
  }
}

template <int G, bool CB, bool DYN>
__global__ void __launch_bounds__(THREADS, G <= 4 ? 3 : 2) attn_kernel(Args a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<G> &sm = *reinterpret_cast<Smem<G> *>(smem_raw);
  // Step form: nothing this kernel reads is written by the query rotation that precedes it except the
  // fragments, which the history consumers load after their wait; the rest (pool counters, page tables,
  // history pages, the window slots the BF16 CTAs read, q) is unchanged until the merge that follows.
  if (!a.step) pdl_wait();
  pdl_trigger();
  const int bid = (int)blockIdx.x;
  const bool is_bf = a.hist_first ? bid >= a.n_hist : bid < a.n_bf;
  if (is_bf)
    part::bf16_role<G>(a, sm, a.hist_first ? bid - a.n_hist : bid, sm.ring[0], [&](int b, int kvh, Smem<G> &, bool &wait) {
      wait = true;  // q_rot is written by the query rotation that precedes this kernel
      return a.qrot + ((size_t)b * a.p.Hq + kvh * G) * D;
    });
  else hist_role<G, CB, DYN>(a, sm, a.hist_first ? bid : bid - a.n_bf);
  // every thread has waited for the query rotation before the grid completes: the merge's wait (and the
  // next step's query rotation, which overwrites the fragments) then follows it as well
  if (a.step) pdl_wait();
}

// ---------------------------------------------------------------------------------------------
// Merge: grid (G, Hkv, B), 512 threads; one CTA per (query head of the group, KV head, sequence).
// The history partials of a segment sit in consecutive slots (CTA index + segment index), the demoted
// token's partial (decode step) and the five BF16 partials in slots of their own.  Latency bound:
// everything that does not depend on the attention kernel's partials is done before the
// griddepcontrol.wait (the partials' location from the pool counters, R_v staged in shared memory), so
// that after it only the partials are read (one round trip per PMAX slots) and combined.  The un-rotation
// o[c] = sum_j o_rot[j] R_v[c][j] gives thread (slice sl, channel c) the 32 terms j = 32 sl .. 32 sl + 31.
// Decode-step form (k_new != NULL): the pool counters still hold the state before the step (every kernel
// of the step read them).  After the wait the CTA of query head 0 stores the new token of its KV head
// into the sink or the window; the CTA that arrives last on pool.sync[0] (each CTA arrives once it has
// read every counter it needs, before its wait) advances every sequence's counters after the wait, so
// no merge CTA reads a counter that this step has already advanced, however many waves the grid takes.
constexpr int MT = 512;
constexpr int RV_LD = D + 4;  // padded row stride of the shared copy of R_v
constexpr int PMAX = 96;      // partial slots staged in shared memory per round
constexpr int PMAX_WIDE = 48; // the same in the wide build (two CTAs per SM)
constexpr uint32_t PART_BYTES = PART_STRIDE * sizeof(float);
__host__ __device__ constexpr size_t merge_smem(bool wide) {
  return (size_t)D * RV_LD * sizeof(float) + (size_t)(wide ? PMAX_WIDE : PMAX) * PART_BYTES;
}
// hpc query heads per CTA (grid G / hpc x Hkv x B): large grids merge several heads of a (sequence, KV head)
// in one CTA, one after the other, with one copy of R_v and one location of the partials; their partials
// are staged together (one round trip) when they fit.  WIDE: the build for grids of more CTAs than SMs, with
// a smaller staging buffer so that two CTAs share an SM.
template <int G, bool WIDE>
__global__ void __launch_bounds__(MT, WIDE ? 2 : 1) merge_kernel(PoolArgs p, const float *part, int n_hist, float *out,
                                                   const uint16_t *k_new, const uint16_t *v_new, int hpc, int dyn) {
  constexpr int PM = WIDE ? PMAX_WIDE : PMAX;
  extern __shared__ float4 rvs4[];  // R_v of this KV head (row stride RV_LD floats), then the staged slots
  float *pst = reinterpret_cast<float *>(rvs4 + D * (RV_LD / 4));
  __shared__ float Osl[4][D], Obs[4][D], Orot[D];
  __shared__ float pw[PM], s_stat[2];
  __shared__ long long s_pref, s_total;
  __shared__ int s_last_all;
  const int kvh = blockIdx.y, b = blockIdx.z, seg = b * p.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = tid & (D - 1), sl = tid >> 7;
  const bool step = k_new != nullptr;
  // R_v rows into shared memory (coalesced 16-byte loads; the wide build in two batches, for its registers)
  {
    const float4 *R4 = reinterpret_cast<const float4 *>(p.R_v + (size_t)kvh * D * D);
    constexpr int NB = WIDE ? 4 : 8;
#pragma unroll
    for (int k0 = 0; k0 < 8; k0 += NB) {
      float4 rv[NB];
#pragma unroll
      for (int k = 0; k < NB; ++k) rv[k] = R4[tid + MT * (k0 + k)];
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        const int i = tid + MT * (k0 + k);
        rvs4[(i / (D / 4)) * (RV_LD / 4) + i % (D / 4)] = rv[k];
      }
    }
  }
  StepState st{};
  if (step) st = step_state(p, b);
  // the partials' location (pool counters, unchanged until the grid's last arrival advances them): the
  // history pages of all sequences and of the sequences before b, from one round of independent loads
  if (warp == 0) {
    long long total = 0, pref = 0;
#pragma unroll 8
    for (int x = lane; x < p.B; x += 32) {
      const long long v = (long long)npages_of(p, x) * p.Hkv;
      total += v;
      if (x < b) pref += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      total += __shfl_xor_sync(FULL, total, o);
      pref += __shfl_xor_sync(FULL, pref, o);
    }
    if (lane == 0) { s_pref = pref; s_total = total; }
  }
  const int np = npages_of(p, b);
  __syncthreads();  // every counter read of this CTA is done
  if (step && tid == 0) {
    __threadfence();
    s_last_all = atomicAdd(p.sync, 1) == (int)(gridDim.x * gridDim.y * gridDim.z) - 1;
  }
  // the segment's pages [start, end): the static ranges' slots i0 + seg .. (nh of them), then the dynamic
  // chunks' slots dyn_slot0 + k0 + seg .. (nd of them)
  int nh = 0, i0 = 0, nd = 0;
  long long k0 = 0;
  if (np > 0) {
    const split::Plan pl = split::plan_of(s_total, n_hist, dyn != 0);
    const long long start = s_pref + (long long)kvh * np, end = start + np;
    const long long send = min(end, pl.static_pages);
    if (start < send) {
      i0 = (int)(start / pl.chunk);
      nh = (int)((send - 1) / pl.chunk) - i0 + 1;
    }
    if (end > pl.static_pages) {
      k0 = (max(start, pl.static_pages) - pl.static_pages) / pl.dyn_pages;
      nd = (int)((end - 1 - pl.static_pages) / pl.dyn_pages - k0 + 1);
    }
  }
  const long long dyn_slot0 = (long long)n_hist + 7LL * p.B * p.Hkv;
  // (the debug build checks the located slots against the workspace's slot ranges)
  if (!OSCAR_DCHECK(nh == 0 || ((long long)i0 + seg + nh <= (long long)n_hist + p.B * p.Hkv && i0 >= 0), p.err)) nh = 0;
  if (!OSCAR_DCHECK(nd == 0 || (k0 + nd <= split::max_dyn_chunks(n_hist) && k0 >= 0), p.err)) nd = 0;
  const int nrot = nh + nd + (step ? 1 : 0);  // rotated-space partials: history (+ the demoted token)
  const int nparts = nrot + 5;
  const size_t stride = (size_t)G * PART_STRIDE;
  __syncthreads();  // s_last_all
  // the grid's last arrival: every sequence's counters after the step (the first MT are read here, while
  // no CTA reads them any more, and kept in registers for the stores after the wait)
  const bool last_all = step && s_last_all;
  StepState sa{};
  if (last_all && tid < p.B) sa = step_state(p, tid);
  pdl_wait();
  pdl_trigger();
  // slot i of the segment (every head's values), i < nparts: history, dynamic chunks, demoted token, BF16
  const float *hp = part + ((size_t)i0 + seg) * stride;
  const float *dp = part + ((size_t)n_hist + (size_t)p.B * p.Hkv * 6 + seg) * stride;
  const float *bp = part + ((size_t)n_hist + (size_t)p.B * p.Hkv + (size_t)seg * 5) * stride;
  const float *yp = part + ((size_t)dyn_slot0 + (size_t)k0 + seg) * stride;
  auto slot = [&](int i) {
    return i < nh ? hp + (size_t)i * stride
           : i < nh + nd ? yp + (size_t)(i - nh) * stride
           : i < nrot ? dp : bp + (size_t)(i - nrot) * stride;
  };
  // Staging: n entries into shared memory by 16-byte loads of every thread (one round trip); entry e holds
  // the PART_STRIDE floats of query head blockIdx.x * hpc + hh of slot i, (hh, i) = at(e).
  constexpr int V4 = PART_STRIDE / 4;  // float4 per staged entry
  auto stage = [&](int n, auto at) {
    constexpr int PER = (PM * V4 + MT - 1) / MT;
    float4 v[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = tid + MT * k;
      if (e < n * V4) {
        const int2 hi = at(e / V4);
        v[k] = reinterpret_cast<const float4 *>(slot(hi.y) + (size_t)(blockIdx.x * hpc + hi.x) * PART_STRIDE)[e % V4];
      }
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = tid + MT * k;
      if (e < n * V4) reinterpret_cast<float4 *>(pst)[e] = v[k];
    }
  };
  // every head's partials in one round when they fit (entry hh * nparts + i)
  const bool together = hpc > 1 && nparts * hpc <= PM;
  if (together) {
    stage(nparts * hpc, [&](int e) { return make_int2(e / nparts, e % nparts); });
    __syncthreads();
  }
  for (int hh = 0; hh < hpc; ++hh) {
  const int h = blockIdx.x * hpc + hh;
  // Rounds of PM staged slots (one round when staged together above); warp 0 forms the round's maximum,
  // the weights and their sum once, and the threads (slice, channel) add the weighted outputs of every
  // fourth slot.  Rounds combine with a running maximum.
  float M = -INFINITY, L = 0.f, acc = 0.f, accb = 0.f;
  for (int r0 = 0; r0 < nparts; r0 += PM) {
    const int n = min(PM, nparts - r0);
    const float *ps = pst;
    if (together) {
      ps = pst + (size_t)hh * nparts * PART_STRIDE;
    } else {
      stage(n, [&](int e) { return make_int2(hh, r0 + e); });
      __syncthreads();
    }
    if (warp == 0) {
      float mr = -INFINITY;
      for (int i = lane; i < n; i += 32) mr = fmaxf(mr, ps[(size_t)i * PART_STRIDE + D]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mr = fmaxf(mr, __shfl_xor_sync(FULL, mr, o));
      const float Mn = fmaxf(M, mr);
      float lr = 0.f;
      for (int i = lane; i < n; i += 32) {
        const float m = ps[(size_t)i * PART_STRIDE + D];
        const float w = m == -INFINITY ? 0.f : exp2f(m - Mn);
        pw[i] = w;
        lr = fmaf(w, ps[(size_t)i * PART_STRIDE + D + 1], lr);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lr += __shfl_xor_sync(FULL, lr, o);
      if (lane == 0) { s_stat[0] = Mn; s_stat[1] = lr; }
    }
    __syncthreads();
    const float Mn = s_stat[0];
    const float f = (M == -INFINITY || Mn == M) ? 1.f : exp2f(M - Mn);  // rescale of the earlier rounds
    L = fmaf(L, f, s_stat[1]);
    acc *= f;
    accb *= f;
    M = Mn;
    for (int i = sl; i < n; i += 4) {  // rotated-space partials and BF16 partials (original space) apart
      const float w = pw[i], o = ps[(size_t)i * PART_STRIDE + ch];
      if (r0 + i < nrot) acc = fmaf(w, o, acc);
      else accb = fmaf(w, o, accb);
    }
    __syncthreads();  // the next round overwrites the staged slots
  }
  Osl[sl][ch] = acc;
  Obs[sl][ch] = accb;
  __syncthreads();
  if (sl == 0) Orot[ch] = ((Osl[0][ch] + Osl[1][ch]) + Osl[2][ch]) + Osl[3][ch];
  __syncthreads();
  {
    const float4 *o4 = reinterpret_cast<const float4 *>(Orot + 32 * sl);
    const float4 *r4 = rvs4 + ch * (RV_LD / 4) + 8 * sl;
    float u0 = 0.f, u1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 o = o4[k], r = r4[k];
      u0 = fmaf(r.x, o.x, fmaf(r.y, o.y, u0));
      u1 = fmaf(r.z, o.z, fmaf(r.w, o.w, u1));
    }
    Osl[sl][ch] = u0 + u1;  // every read of Osl finished before the barrier above
  }
  __syncthreads();
  if (sl == 0) {
    const float o = (((Osl[0][ch] + Osl[1][ch]) + Osl[2][ch]) + Osl[3][ch]) +
                    (((Obs[0][ch] + Obs[1][ch]) + Obs[2][ch]) + Obs[3][ch]);
    out[((size_t)b * p.Hq + kvh * G + h) * D + ch] = L > 0.f ? o / L : 0.f;
  }
  __syncthreads();  // the next head reuses Osl, Obs and Orot
  }
  if (!step) return;
  if (blockIdx.x == 0 && st.append && tid < 2 * (D / 4)) {  // the new token of KV head kvh (8-byte pieces of K and V)
    const int kv = tid / (D / 4), j = tid % (D / 4);
    uint16_t *dst = st.to_sink
        ? (kv == 0 ? p.sink_k : p.sink_v) + (((size_t)b * p.Hkv + kvh) * SINK + st.slen) * D
        : (kv == 0 ? p.recent_k : p.recent_v) + (((size_t)b * p.Hkv + kvh) * RECENT + (st.nrs + st.nrl - 1) % RECENT) * D;
    reinterpret_cast<uint2 *>(dst)[j] = reinterpret_cast<const uint2 *>((kv == 0 ? k_new : v_new) + ((size_t)b * p.Hkv + kvh) * D)[j];
  }
  if (last_all) {
    for (int bb = tid; bb < p.B; bb += MT) {
      const StepState s2 = bb < MT ? sa : step_state(p, bb);
      if (!s2.ok) atomicOr(p.err, OSCAR_DEVERR_COUNTERS);
      else if (s2.want && !s2.demote)
        atomicOr(p.err, s2.hl / PAGE >= p.max_pages ? OSCAR_DEVERR_HISTORY_FULL : OSCAR_DEVERR_PAGE_INDEX);
      if (s2.ok && (s2.demote || s2.append)) {
        p.sink_len[bb] = s2.nslen;
        p.hist_len[bb] = s2.nhl;
        p.recent_start[bb] = s2.nrs;
        p.recent_len[bb] = s2.nrl;
      }
    }
    if (tid == 0) p.sync[0] = 0;
  }
}

}  // namespace v1

// ---------------------------------------------------------------------------------------------
// Grid of the attention kernel: BF16 CTAs (5 per sequence and KV head) first, then history CTAs
// sized so that both fit in one wave of resident CTAs (history CTAs get at least 5/6 of it; when the BF16
// CTAs outnumber the rest they run in waves in the remaining sixth, alongside the history CTAs: measured
// on the 32k batch sweep, a quarter left the history CTAs too few slots and an eighth gained nothing more).
constexpr int BF_SHARE = 6;
template <int G, bool CB>
static int resident_ctas() {
  static std::atomic<int> slots[kMaxDevices];
  return per_device(slots, [](int dev) {
    int sms = 148, occ = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = (int)sizeof(v1::Smem<G>);
    cudaFuncSetAttribute(v1::attn_kernel<G, CB, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v1::attn_kernel<G, CB, false>, v1::THREADS, smem) != cudaSuccess ||
        occ < 1)
      occ = 1;
    return sms * occ;
  });
}

template <bool CB>
static int resident_ctas_for(int G) {
  switch (G) {
    case 1: return resident_ctas<1, CB>();
    case 2: return resident_ctas<2, CB>();
    case 4: return resident_ctas<4, CB>();
    default: return resident_ctas<8, CB>();
  }
}

// Pools with a codebook for K or V run the codebook form of the attention kernel.
static bool has_codebook(const PoolArgs &p) { return p.cb_k != nullptr || p.cb_v != nullptr; }

int v1_hist_ctas(const PoolArgs &p) {
  const int slots = has_codebook(p) ? resident_ctas_for<true>(p.Hq / p.Hkv) : resident_ctas_for<false>(p.Hq / p.Hkv);
  const long long nbf = (long long)p.B * p.Hkv * 5;
  long long n = slots - (nbf < slots / BF_SHARE ? nbf : slots / BF_SHARE);
  if (n > 1000) n = 1000;
  const long long cap = (long long)p.B * p.Hkv * p.max_pages;
  if (cap < n) n = cap;
  return (int)(n < 1 ? 1 : n);
}

// Partial slots: history (CTA index + segment index), 5 BF16 and one demoted-token slot per segment, then
// (dynamic tail) chunk index + segment index.
static size_t v1_slots(const PoolArgs &p, bool dyn) {
  const int nh = v1_hist_ctas(p);
  return (size_t)nh + (size_t)p.B * p.Hkv * 7 + (dyn ? (size_t)split::max_dyn_chunks(nh) + (size_t)p.B * p.Hkv : 0);
}
size_t v1_ws_bytes(const PoolArgs &p, bool dyn) {
  const int G = p.Hq / p.Hkv;
  const size_t frag = (size_t)p.B * p.Hkv * (G > 4 ? 36 : 18) * 32 * sizeof(uint32_t);
  return (size_t)p.B * p.Hq * D * sizeof(float) + frag + v1_slots(p, dyn) * G * PART_STRIDE * sizeof(float) +
         (dyn ? 16 : 0);
}

// Workspace: [q_rot][query fragments][partial slots].  k_new != NULL: the decode-step form.
template <int G>
static cudaError_t launch_v1_g(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                               cudaStream_t s, bool dyn, const uint16_t *k_new = nullptr,
                               const uint16_t *v_new = nullptr) {
  v1::Args a;
  a.p = p;
  a.q = q;
  a.qrot = ws;
  uint32_t *frag = reinterpret_cast<uint32_t *>(ws + (size_t)p.B * p.Hq * D);
  a.frag = frag;
  a.part = reinterpret_cast<float *>(frag + (size_t)p.B * p.Hkv * v1::frag_words<G>() * 32);
  a.sm_log2 = sm_scale * 1.4426950408889634f;
  a.n_hist = v1_hist_ctas(p);
  // the dynamic tail only where the pool can hold 64 history pages per history CTA (split::plan_of)
  dyn = dyn && (long long)p.B * p.Hkv * p.max_pages >= 64LL * a.n_hist;
  a.dyn = dyn ? 1 : 0;
  a.dyn_ctr = dyn ? reinterpret_cast<unsigned long long *>(a.part + v1_slots(p, true) * G * PART_STRIDE) : nullptr;
  const int nbf = p.B * p.Hkv * 5;
  a.n_bf = nbf;
  {
    const int slots = has_codebook(p) ? resident_ctas_for<true>(G) : resident_ctas_for<false>(G);
    a.hist_first = nbf > slots / BF_SHARE ? 1 : 0;
  }
  const int smem = (int)sizeof(v1::Smem<G>);
  auto attn = has_codebook(p) ? (dyn ? v1::attn_kernel<G, true, true> : v1::attn_kernel<G, true, false>)
                              : (dyn ? v1::attn_kernel<G, false, true> : v1::attn_kernel<G, false, false>);
  cudaError_t e = cudaFuncSetAttribute(attn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  a.step = k_new != nullptr;
  a.k_new = k_new;
  a.v_new = v_new;
  // Step form: the attention reads only state the step leaves unchanged and its BF16 CTAs perform the
  // demotion (overlapping the history CTAs); the merge performs the append and the counter update.
  if ((e = launch_pdl(v1::qrot_kernel<G>, dim3(p.B * p.Hkv), dim3(512), 0, s, p, q, ws, frag, a.sm_log2, a.dyn_ctr)) !=
      cudaSuccess)
    return e;
  profile_begin(OSCAR_PROFILE_HISTORY, s);
  if ((e = launch_pdl(attn, dim3(a.n_hist + nbf), dim3(v1::THREADS), smem, s, a)) != cudaSuccess) return e;
  profile_end(OSCAR_PROFILE_HISTORY, s);
  return launch_merge_v1(p, (const float *)a.part, a.n_hist, out, k_new, v_new, s, dyn);
}

// The merge of a decode launch whose partial slots follow this file's layout (history slots cta + segment
// for n_hist history CTAs, then the BF16 and demoted-token slots); k_new != NULL: the decode-step form.
// Merge grid: grids of more CTAs than SMs run the wide build (two CTAs per SM); query heads per CTA: the
// smallest power of two (at most G) that brings the grid within one wave of it, or, past G, as many waves as
// it takes.
static int merge_sms(const PoolArgs &) {
  static std::atomic<int> sms_cache[kMaxDevices];
  return per_device(sms_cache, [](int dev) {
    int n = 148;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
  });
}
static int merge_heads_per_cta(const PoolArgs &p) {
  const int sms = merge_sms(p), G = p.Hq / p.Hkv;
  int hpc = 1;
  while (hpc < G && (long long)(G / hpc) * p.Hkv * p.B > 2LL * sms) hpc *= 2;
  return hpc;
}

cudaError_t launch_merge_v1(const PoolArgs &p, const float *part, int n_hist, float *out, const uint16_t *k_new,
                            const uint16_t *v_new, cudaStream_t s, bool dyn) {
  const int hpc = merge_heads_per_cta(p);
  const bool wide = (long long)(p.Hq / p.Hkv / hpc) * p.Hkv * p.B > merge_sms(p);
  const size_t smem = v1::merge_smem(wide);
  auto go = [&](auto kernel) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(p.Hq / p.Hkv / hpc, p.Hkv, p.B), dim3(v1::MT), smem, s, p, part, n_hist, out,
                      k_new, v_new, hpc, dyn ? 1 : 0);
  };
  switch (p.Hq / p.Hkv) {
    case 1: return wide ? go(v1::merge_kernel<1, true>) : go(v1::merge_kernel<1, false>);
    case 2: return wide ? go(v1::merge_kernel<2, true>) : go(v1::merge_kernel<2, false>);
    case 4: return wide ? go(v1::merge_kernel<4, true>) : go(v1::merge_kernel<4, false>);
    case 8: return wide ? go(v1::merge_kernel<8, true>) : go(v1::merge_kernel<8, false>);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_v1(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                             cudaStream_t s, bool dyn) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_v1_g<1>(p, q, out, sm_scale, ws, s, dyn);
    case 2: return launch_v1_g<2>(p, q, out, sm_scale, ws, s, dyn);
    case 4: return launch_v1_g<4>(p, q, out, sm_scale, ws, s, dyn);
    case 8: return launch_v1_g<8>(p, q, out, sm_scale, ws, s, dyn);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_step_v1(const PoolArgs &p, const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q,
                           float *out, float sm_scale, float *ws, cudaStream_t s, bool dyn) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_v1_g<1>(p, q, out, sm_scale, ws, s, dyn, k_new, v_new);
    case 2: return launch_v1_g<2>(p, q, out, sm_scale, ws, s, dyn, k_new, v_new);
    case 4: return launch_v1_g<4>(p, q, out, sm_scale, ws, s, dyn, k_new, v_new);
    case 8: return launch_v1_g<8>(p, q, out, sm_scale, ws, s, dyn, k_new, v_new);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oscar

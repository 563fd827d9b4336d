// Decode attention over the three-segment pool, tensor-core version (group size 128).
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": the INT2 kernel
// unpacks the 2-bit codes, dequantizes with scale/zero point and accumulates in floating point; a
// BF16 kernel handles the sink and recent window; an online-softmax merge combines the results.
// "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract: a
// custom INT2 attention kernel compatible with paged KV-cache serving.
//
// Three launches:
//   qrot_kernel   q_rot = q · R_k for every query head (row-vector convention), fp32.
//   attn_kernel   BF16 CTAs (first block indices): 64 sink or recent tokens each, plain FMA, one
//                 partial per chunk.  History CTAs: the flattened (sequence, KV head, page) space is
//                 cut into equal contiguous ranges, one per CTA; a producer warp streams up to two
//                 pages of one segment per ring stage (codes and scale/zero rows) into shared memory
//                 with 1-D bulk async copies; four consumer warps each score one 16-token tile of
//                 every page of the stage with warp MMAs (m16n8k16, f16 inputs, f32 accumulate) and
//                 accumulate P·V the same way, with a lazily rescaled online softmax; one
//                 (m, l, o_rot) partial per head is written per (CTA, segment).
//   merge_kernel  LSE-combines a segment's partials, un-rotates the history part (o · R_v^T),
//                 adds the BF16 part and normalises.
//
// Exactness of the tensor-core arithmetic: a 2-bit code c placed in the low mantissa bits of an
// fp16 with a zero exponent field is the subnormal c * 4^k * 2^-24 (k = its bit position / 2), so
// codes enter the MMA exactly with one AND per two codes.  q_rot and the softmax weights are split
// into two fp16 terms (hi + lo, 22 significant bits), pre-scaled by powers of two (including 4^-k)
// so that fp16 holds them; scale and zero point are applied in fp32 outside the MMA:
//   score = scale * sum_c code_c q_c + zero * sum_c q_c,   o_rot = sum_t p_t scale_t code_t + sum_t p_t zero_t.
// Softmax values are kept in base 2 (scores pre-multiplied by log2 e), so partials carry log2 maxima.
#include "oscar_internal.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {

namespace v1 {

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
  const float *qrot;   // [B][Hq][D]
  const uint16_t *q;   // [B][Hq][D] bf16
  float sm_log2;       // softmax_scale * log2(e)
  int n_hist;          // history CTAs (block indices n_bf .. n_bf + n_hist - 1)
  int n_bf;            // BF16 CTAs (block indices 0 .. n_bf - 1)
  float *part;         // partial slots [*][G][PART_STRIDE]
};

__device__ __forceinline__ int npages_of(const PoolArgs &p, int b) {
  int hl = p.hist_len[b];
  hl = max(0, min(hl, p.max_pages * PAGE));
  return (hl + PAGE - 1) / PAGE;
}

// Unpack one 32-bit word of 16 codes (code j at bits 2j) into 8 fp16x2 registers at r[base..base+7]:
// register k holds (code k, code 8+k) as fp16 subnormals scaled by 4^k (k <= 4) or 4^(k-5) (k >= 5).
__device__ __forceinline__ void unpack16(uint32_t x, uint32_t (&r)[16], int base) {
#pragma unroll
  for (int k = 0; k < 5; ++k) r[base + k] = x & (0x00030003u << (2 * k));
  const uint32_t xs = x >> 10;
#pragma unroll
  for (int k = 0; k < 3; ++k) r[base + 5 + k] = xs & (0x00030003u << (2 * k));
}
__device__ __forceinline__ float code_factor_inv(int k) {  // 1 / 4^k' for register k (0..7)
  const int e = (k <= 4) ? 2 * k : 2 * (k - 5);
  return __int_as_float((127 - e) << 23);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }

// Map a flattened page index to (b, kvh, local page) by a warp-cooperative scan over sequences.
// Run by one full warp; results valid in every lane.  total receives the number of pages.
__device__ void locate(const PoolArgs &p, long long start, int &b0, int &kvh0, int &local0, long long &total) {
  const int lane = threadIdx.x & 31;
  long long run = 0;
  b0 = -1; kvh0 = 0; local0 = 0;
  for (int base = 0; base < p.B; base += 32) {
    const int b = base + lane;
    const long long v = (b < p.B) ? (long long)npages_of(p, b) * p.Hkv : 0;
    long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += t;
    }
    const long long excl = run + inc - v;
    const unsigned hit = __ballot_sync(FULL, b < p.B && v > 0 && start >= excl && start < excl + v);
    if (b0 < 0 && hit) {
      const int src = __ffs(hit) - 1;
      const long long e = __shfl_sync(FULL, excl, src);
      const int bb = base + src;
      const int np = npages_of(p, bb);
      b0 = bb;
      kvh0 = (int)((start - e) / np);
      local0 = (int)((start - e) % np);
    }
    run += __shfl_sync(FULL, inc, 31);
  }
  total = run;
}

// This CTA's share of the flattened (sequence, KV head, page) space: pages [lo, lo + n) with
// chunk = ceil(total / n_hist), lo = cta * chunk, and the position (b0, kvh0, local0) of page lo plus
// the page count np0 and history length hl0 of sequence b0.  Run by one full warp; results valid in
// every lane.  Up to 32 sequences one load of hist_len per lane serves everything.
__device__ void locate_range(const PoolArgs &p, int n_hist, int cta, long long &lo, long long &n, int &b0, int &kvh0,
                             int &local0, int &np0, int &hl0) {
  const int lane = threadIdx.x & 31;
  b0 = 0; kvh0 = 0; local0 = 0; np0 = 0; hl0 = 0;
  if (p.B <= 32) {
    const int hl = lane < p.B ? max(0, min(p.hist_len[lane], p.max_pages * PAGE)) : 0;
    const int np = (hl + PAGE - 1) / PAGE;
    const long long v = (long long)np * p.Hkv;
    long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += t;
    }
    const long long total = __shfl_sync(FULL, inc, 31);
    const long long chunk = (total + n_hist - 1) / n_hist;
    lo = (long long)cta * chunk;
    n = max(0ll, min(total, lo + chunk) - lo);
    const long long excl = inc - v;
    const unsigned hit = __ballot_sync(FULL, v > 0 && lo >= excl && lo < excl + v);
    if (n > 0 && hit) {
      const int src = __ffs(hit) - 1;
      const long long e = __shfl_sync(FULL, excl, src);
      np0 = __shfl_sync(FULL, np, src);
      hl0 = __shfl_sync(FULL, hl, src);
      b0 = src;
      kvh0 = (int)((lo - e) / np0);
      local0 = (int)((lo - e) % np0);
    }
    return;
  }
  long long total;
  locate(p, 0, b0, kvh0, local0, total);  // total only
  const long long chunk = (total + n_hist - 1) / n_hist;
  lo = (long long)cta * chunk;
  n = max(0ll, min(total, lo + chunk) - lo);
  if (n > 0) {
    locate(p, lo, b0, kvh0, local0, total);
    np0 = npages_of(p, b0);
    hl0 = max(0, min(p.hist_len[b0], p.max_pages * PAGE));
  }
}

template <int G>
struct Smem {
  static constexpr int NT = (2 * G + 7) / 8;
  alignas(128) uint8_t ring[NSTAGE][STAGE_BYTES];
  uint64_t full[NSTAGE][STAGE_PAGES], empty[NSTAGE][STAGE_PAGES];  // one pair per page slot
  uint64_t csync;                                                    // consumer-warp barrier
  int meta_seg[NSTAGE], meta_ntok[NSTAGE][STAGE_PAGES], meta_flags[NSTAGE];  // flags: 1 last, 2 abort
  float qr[G][D];
  float kfac[G], zfac[G];
  int sigma[G];
  float wm[CONSUMER_WARPS][G], wl[CONSUMER_WARPS][G], wz[CONSUMER_WARPS][G];
  float wo[CONSUMER_WARPS][G][D];
  float pbuf[CONSUMER_WARPS][G][16];
  long long range_lo, range_n;
  int b0, kvh0, local0, np0, hl0;
};

// ---------------------------------------------------------------------------------------------
// q_rot = q . R_k for the G query heads of one (sequence, KV head): grid B * Hkv, 512 threads; thread
// (c, quarter) sums rows 16k .. 16k+15 for k = 2 quarter, 2 quarter + 1 of column c, and the eight
// partial sums are added as ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7)) — the order the demotion
// kernel uses when it rotates the queries in oscar_decode_step, so both paths give the same bits.
template <int G>
__global__ void __launch_bounds__(512) qrot_kernel(PoolArgs p, const uint16_t *q, float *qrot) {
  __shared__ float qs[G][D];
  __shared__ float part[8][G][D];
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x, b = s / p.Hkv, kvh = s % p.Hkv;
  const int tid = threadIdx.x, c = tid & (D - 1), qt = tid >> 7;
  for (int i = tid; i < G * D; i += 512) qs[i / D][i % D] = bf16_to_f32(q[((size_t)b * p.Hq + kvh * G) * D + i]);
  const float *R = p.R_k + (size_t)kvh * D * D + (size_t)(32 * qt) * D + c;
  float r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = R[(size_t)i * D];
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
    for (int h = 0; h < G; ++h)
      qrot[((size_t)b * p.Hq + kvh * G + h) * D + c] =
          ((part[0][h][c] + part[1][h][c]) + (part[2][h][c] + part[3][h][c])) +
          ((part[4][h][c] + part[5][h][c]) + (part[6][h][c] + part[7][h][c]));
}

// ---------------------------------------------------------------------------------------------
// BF16 sink/recent chunk: block index = segment * 5 + chunk (chunk 0 = sink, 1..4 = recent tokens
// 64(chunk-1) .. 64 chunk - 1 counted from the oldest).
template <int G>
__device__ __forceinline__ void bf16_role(const Args &a, Smem<G> &sm) {
  const PoolArgs &p = a.p;
  const int idx = blockIdx.x;
  const int seg = idx / 5, chunk = idx % 5, b = seg / p.Hkv, kvh = seg % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float *slot = a.part + ((size_t)a.n_hist + (size_t)p.B * p.Hkv + (size_t)seg * 5 + chunk) * G * PART_STRIDE;
  if (warp >= CONSUMER_WARPS) return;
  int slen = p.sink_len[b], rs = p.recent_start[b], rl = p.recent_len[b];
  slen = max(0, min(slen, SINK)); rs = max(0, min(rs, RECENT - 1)); rl = max(0, min(rl, RECENT));
  const int n = (chunk == 0) ? slen : max(0, min(64, rl - (chunk - 1) * 64));
  for (int i = tid; i < G * D; i += 128) sm.qr[i / D][i % D] = bf16_to_f32(a.q[((size_t)b * p.Hq + kvh * G) * D + i]);
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
  const uint16_t *kb = chunk == 0 ? p.sink_k + ((size_t)b * p.Hkv + kvh) * SINK * D
                                  : p.recent_k + ((size_t)b * p.Hkv + kvh) * RECENT * D;
  const uint16_t *vb = chunk == 0 ? p.sink_v + ((size_t)b * p.Hkv + kvh) * SINK * D
                                  : p.recent_v + ((size_t)b * p.Hkv + kvh) * RECENT * D;
  auto row_of = [&](int i) { return chunk == 0 ? i : (rs + (chunk - 1) * 64 + i) % RECENT; };
  // QK: lane -> token (lane & 15) of this warp's 16, channel half (lane >> 4)
  const int tk = 16 * warp + (lane & 15), hf = lane >> 4;
  const bool valid = tk < n;
  float dot[G];
#pragma unroll
  for (int h = 0; h < G; ++h) dot[h] = 0.f;
  if (valid) {
    const uint4 *kr = reinterpret_cast<const uint4 *>(kb + (size_t)row_of(tk) * D + hf * 64);
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = kr[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float kv = bf16_to_f32((ws[e >> 1] >> (16 * (e & 1))) & 0xffffu);
        const int c = hf * 64 + 8 * i + e;
#pragma unroll
        for (int h = 0; h < G; ++h) dot[h] = fmaf(kv, sm.qr[h][c], dot[h]);
      }
    }
  }
  float m2[G], l[G], o[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    dot[h] += __shfl_xor_sync(FULL, dot[h], 16);
    const float s2 = valid ? dot[h] * a.sm_log2 : -INFINITY;
    float mx = s2;
#pragma unroll
    for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o2));
    const float pr = (s2 == -INFINITY) ? 0.f : exp2f(s2 - mx);
    float sum = pr;
#pragma unroll
    for (int o2 = 1; o2 < 16; o2 <<= 1) sum += __shfl_xor_sync(FULL, sum, o2);
    m2[h] = mx; l[h] = sum;
    if (lane < 16) sm.pbuf[warp][h][lane] = pr;
#pragma unroll
    for (int k = 0; k < 4; ++k) o[h][k] = 0.f;
  }
  __syncwarp();
  // PV: lane -> channels 4*lane .. 4*lane+3
  uint2 vv[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int t2 = 16 * warp + j;
    vv[j] = t2 < n ? reinterpret_cast<const uint2 *>(vb + (size_t)row_of(t2) * D)[lane] : make_uint2(0, 0);
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float v[4] = {bf16_to_f32(vv[j].x & 0xffffu), bf16_to_f32(vv[j].x >> 16), bf16_to_f32(vv[j].y & 0xffffu),
                        bf16_to_f32(vv[j].y >> 16)};
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float pj = sm.pbuf[warp][h][j];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[h][k] = fmaf(pj, v[k], o[h][k]);
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) { sm.wm[warp][h] = m2[h]; sm.wl[warp][h] = l[h]; }
#pragma unroll
    for (int k = 0; k < 4; ++k) sm.wo[warp][h][4 * lane + k] = o[h][k];
  }
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
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
        O += e * sm.wo[w][h][tid];
      }
    }
    slot[h * PART_STRIDE + tid] = O;
    if (tid == 0) { slot[h * PART_STRIDE + D] = M; slot[h * PART_STRIDE + D + 1] = L; }
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
template <int G>
__device__ __forceinline__ void setup_segment(const Args &a, Smem<G> &sm, int b, int kvh,
                                              uint32_t (&bq)[Smem<G>::NT][8][2], uint32_t &par) {
  constexpr int NT = Smem<G>::NT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float *src = a.qrot + ((size_t)b * a.p.Hq + kvh * G) * D;
  for (int i = tid; i < G * D; i += 128) sm.qr[i / D][i % D] = src[i];
  consumer_sync(sm, par, a.p.err);
  for (int h = warp; h < G; h += CONSUMER_WARPS) {
    float amax = 0.f, sum = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float v = sm.qr[h][lane + 32 * k];
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
      sm.sigma[h] = sig;
      sm.kfac[h] = pow2f(24 - sig) * a.sm_log2;
      sm.zfac[h] = sum * a.sm_log2;
    }
  }
  consumer_sync(sm, par, a.p.err);
  const int gq = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 4 * nt + (gq >> 1), split = gq & 1;
    const bool live = h < G;
    const float s2 = live ? pow2f(sm.sigma[h]) : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int i = 2 * j + hb;             // register index of the token's 16 (word i/8, slot i%8)
        const int wi = i >> 3, k = i & 7;
        const int ch_lo = 32 * t + 16 * wi + k, ch_hi = ch_lo + 8;
        const float f = code_factor_inv(k) * s2;
        float v[2];
        const int chs[2] = {ch_lo, ch_hi};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x = live ? sm.qr[h][chs[e]] * f : 0.f;
          const float hi = __half2float(__float2half_rn(x));
          v[e] = split == 0 ? hi : x - hi;
        }
        bq[nt][j][hb] = pack_half2(v[0], v[1]);
      }
    }
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

// One page in one consumer warp: all 64 tokens (four 16-token tiles); ntok = valid tokens (1..64).
// Lane (g, t) owns the rows g + 8j (j = 0..7: tile j/2, row half j%2) of the QK accumulators for head
// column t; the softmax weights are formed in that layout, split into fp16 hi + lo and transposed
// with movmatrix into the B operand of the P.V products, whose A operand pairs tokens (2t, 2t+1).
template <int G, bool FULL>
__device__ __forceinline__ void page_pass(const uint8_t *pb, int ntok, const Smem<G> &sm, WarpState<G> &ws,
                                          const uint32_t (&bq)[Smem<G>::NT][8][2]) {
  constexpr int NT = Smem<G>::NT;
  constexpr bool ALL_LIVE = (G % 4) == 0;
  const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
  // ---- QK: A = K codes (tokens 16mt + g, 16mt + g + 8; lane t owns channels 32t .. 32t+31) ----
  float S[4][NT][4];
  const uint8_t *kc = pb + OFF_KC + gq * 32 + 8 * t;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) S[mt][nt][0] = S[mt][nt][1] = S[mt][nt][2] = S[mt][nt][3] = 0.f;
    if (FULL || 16 * mt < ntok) {
      const uint2 ka = *reinterpret_cast<const uint2 *>(kc + (16 * mt) * 32);
      const uint2 kb = *reinterpret_cast<const uint2 *>(kc + (16 * mt + 8) * 32);
      uint32_t T0[16], T1[16];
      unpack16(ka.x, T0, 0); unpack16(ka.y, T0, 8);
      unpack16(kb.x, T1, 0); unpack16(kb.y, T1, 8);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mma16816(S[mt][nt], T0[2 * j], T1[2 * j], T0[2 * j + 1], T1[2 * j + 1], bq[nt][j][0], bq[nt][j][1]);
    }
  }
  // ---- per-row scale / zero of the lane's 8 rows ----
  const uint16_t *Ks = reinterpret_cast<const uint16_t *>(pb + OFF_KS) + gq;
  const uint16_t *Kz = reinterpret_cast<const uint16_t *>(pb + OFF_KZ) + gq;
  const uint16_t *Vs = reinterpret_cast<const uint16_t *>(pb + OFF_VS) + gq;
  const uint16_t *Vz = reinterpret_cast<const uint16_t *>(pb + OFF_VZ) + gq;
  float ks[8], kz[8], vs[8], vz[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool valid = FULL || gq + 8 * j < ntok;
    ks[j] = bf16_to_f32(Ks[8 * j]);
    kz[j] = bf16_to_f32(Kz[8 * j]);
    vs[j] = valid ? bf16_to_f32(Vs[8 * j]) : 0.f;
    vz[j] = valid ? bf16_to_f32(Vz[8 * j]) : 0.f;
  }
  // ---- weight scaling exponent tau: weights p * vs * 2^tau stay below 2^14 ----
  float vmax = fmaxf(max3f(vs[0], vs[1], vs[2]), max3f(max3f(vs[3], vs[4], vs[5]), vs[6], vs[7]));
  vmax = fmaxf(vmax, __shfl_xor_sync(FULL, vmax, 4));
  vmax = fmaxf(vmax, __shfl_xor_sync(FULL, vmax, 8));
  vmax = fmaxf(vmax, __shfl_xor_sync(FULL, vmax, 16));
  if (vmax >= ws.tau_lim && vmax > 0.f) {
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
  uint32_t bw[NT][4][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = ALL_LIVE ? 4 * nt + t : min(4 * nt + t, G - 1);
    const bool live_h = ALL_LIVE || 4 * nt + t < G;
    const float kf = sm.kfac[h], zf = sm.zfac[h];
    float sc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int mt = j >> 1, e = j & 1;
      sc[j] = (FULL || gq + 8 * j < ntok) ? fmaf((S[mt][nt][2 * e] + S[mt][nt][2 * e + 1]) * ks[j], kf, kz[j] * zf)
                                          : -INFINITY;
    }
    float tmax = fmaxf(max3f(sc[0], sc[1], sc[2]), max3f(max3f(sc[3], sc[4], sc[5]), sc[6], sc[7]));
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
    // p * 2^tau = exp2(score - (m - tau)); l and the zero-point sum take p itself
    const float mref = ws.m2[nt] - (float)ws.tau;
    float lsum = 0.f, zsum = 0.f;
    uint32_t wp[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float pr = fast_exp2(sc[j] - mref);  // 0 for rows past ntok (score -inf)
      lsum += pr;
      zsum = fmaf(pr, vz[j], zsum);
      const float w = live_h ? pr * vs[j] : 0.f;
      const __half hh = __float2half_rn(w);
      wp[j] = pack_half2(__half2float(hh), w - __half2float(hh));  // (hi, lo)
    }
    ws.l[nt] = fmaf(lsum, untau, ws.l[nt]);
    ws.oz[nt] = fmaf(zsum, untau, ws.oz[nt]);
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      bw[nt][mt][0] = movmatrix_trans(wp[2 * mt]);
      bw[nt][mt][1] = movmatrix_trans(wp[2 * mt + 1]);
    }
  }
  // ---- P.V per tile: A = V codes^T (tokens 2t, 2t+1 | 2t+8, 2t+9; group g: channels 16g .. 16g+15) ----
  const uint32_t *vrow = reinterpret_cast<const uint32_t *>(pb + OFF_VC) + gq + 2 * t * 8;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    if (!(FULL || 16 * mt < ntok)) continue;
    const uint32_t *vr = vrow + 16 * mt * 8;
    const uint32_t xa = vr[0], xb = vr[8], xc = vr[64], xd = vr[72];
    uint32_t VA[16], VB[16];
    unpack16(prmt(xa, xb, 0x5410), VA, 0); unpack16(prmt(xa, xb, 0x7632), VA, 8);
    unpack16(prmt(xc, xd, 0x5410), VB, 0); unpack16(prmt(xc, xd, 0x7632), VB, 8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int m8 = 0; m8 < 8; ++m8)
        mma16816(ws.O[nt][m8], VA[2 * m8], VA[2 * m8 + 1], VB[2 * m8], VB[2 * m8 + 1], bw[nt][mt][0], bw[nt][mt][1]);
  }
}

template <int G>
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
  if (warp == CONSUMER_WARPS) {  // the producer warp locates this CTA's range
    long long lo, n;
    int b0, kvh0, local0, np0, hl0;
    locate_range(p, a.n_hist, cta, lo, n, b0, kvh0, local0, np0, hl0);
    if (lane == 0) {
      sm.range_lo = lo; sm.range_n = n; sm.b0 = b0; sm.kvh0 = kvh0; sm.local0 = local0; sm.np0 = np0; sm.hl0 = hl0;
    }
  }
  __syncthreads();
  const long long n = sm.range_n;
  if (n <= 0) return;

  if (warp == CONSUMER_WARPS) {
    // ---------------- producer warp: up to STAGE_PAGES pages of one segment per stage ----------------
    // Lane i owns page i of a stage: the page-table entries of a stage are read in one round trip and
    // each lane issues its own page's bulk copies.  hist_len is read once per sequence.
    int b = sm.b0, kvh = sm.kvh0, local = sm.local0;
    int np = sm.np0, hl = sm.hl0;
    int stage = 0, it = 0;
    uint32_t phase = 0;
    long long done = 0;
    while (done < n) {
      bool abort = false;
      if (it >= NSTAGE) {  // every page slot of the stage released by its consumer warp
        bool okw = true;
        if (lane < STAGE_PAGES) okw = mbar_wait_bounded(&sm.empty[stage][lane], phase ^ 1);
        abort = !__all_sync(FULL, okw);
        if (abort && lane == 0) atomicOr(p.err, OSCAR_DEVERR_TIMEOUT);
      }
      const int seg = b * p.Hkv + kvh;
      const int cnt = abort ? 0 : (int)min((long long)STAGE_PAGES, min(n - done, (long long)(np - local)));
      int pp = -1, ntk = 0;
      if (lane < cnt) {
        const int lp = local + lane;
        pp = p.page_table[(size_t)b * p.max_pages + lp];
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
        sm.meta_flags[stage] = (done + cnt >= n ? 1 : 0) | (abort ? 2 : 0);
      }
      __syncwarp();  // the stage's metadata is written before any of its slots can complete
      if (lane < STAGE_PAGES) {
        uint64_t *bar = &sm.full[stage][lane];
        if (have) {
          mbar_arrive_expect_tx(bar, (uint32_t)PAGE_BYTES);
          uint8_t *dst = sm.ring[stage] + lane * PAGE_BYTES;
          const size_t row = ((size_t)pp * p.Hkv + kvh) * PAGE;
          bulk_g2s(dst + OFF_KC, p.codes_k + row * (D / 4), 2048, bar);
          bulk_g2s(dst + OFF_VC, p.codes_v + row * (D / 4), 2048, bar);
          bulk_g2s(dst + OFF_KS, p.scale_k + row, 128, bar);
          bulk_g2s(dst + OFF_KZ, p.zero_k + row, 128, bar);
          bulk_g2s(dst + OFF_VS, p.scale_v + row, 128, bar);
          bulk_g2s(dst + OFF_VZ, p.zero_v + row, 128, bar);
        } else {
          mbar_arrive(bar);
        }
      }
      if (abort) {
        // wait (bounded) for the copies still in flight into stages the consumers may not read
        if (lane < STAGE_PAGES)
          for (int k = max(0, it - NSTAGE + 1); k < it; ++k)
            mbar_wait_bounded(&sm.full[k % NSTAGE][lane], (uint32_t)((k / NSTAGE) & 1));
        break;
      }
      done += cnt;
      local += cnt;
      if (local == np && done < n) {
        local = 0;
        if (++kvh == p.Hkv) {
          kvh = 0;
          do { ++b; } while (b < p.B && npages_of(p, b) == 0);
          if (b < p.B) {
            np = npages_of(p, b);
            hl = max(0, min(p.hist_len[b], p.max_pages * PAGE));
          }
        }
      }
      ++it;
      if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
    }
    return;
  }
  // ---------------- consumers ----------------
  WarpState<G> ws;
  reset(ws);
  uint32_t bq[NT][8][2];
  // the first segment's query setup needs no pages: it overlaps the first bulk copies
  int cur = sm.b0 * p.Hkv + sm.kvh0, stage = 0;
  ws.csync_par = 0;
  setup_segment(a, sm, sm.b0, sm.kvh0, bq, ws.csync_par);
  uint32_t phase = 0;
  while (true) {
    if (!mbar_wait_bounded(&sm.full[stage][warp], phase)) {
      if (lane == 0) atomicOr(a.p.err, OSCAR_DEVERR_TIMEOUT);
      break;
    }
    const int flags = sm.meta_flags[stage];
    if (flags & 2) break;  // producer aborted
    const int seg = sm.meta_seg[stage];
    if (seg != cur) {
      if (cur >= 0) flush(a, sm, ws, a.part + ((size_t)cta + cur) * G * PART_STRIDE);
      cur = seg;
      setup_segment(a, sm, seg / p.Hkv, seg % p.Hkv, bq, ws.csync_par);
    }
    const int ntok = sm.meta_ntok[stage][warp];
    const uint8_t *pb = sm.ring[stage] + warp * PAGE_BYTES;
    if (ntok == PAGE) page_pass<G, true>(pb, ntok, sm, ws, bq);
    else if (ntok > 0) page_pass<G, false>(pb, ntok, sm, ws, bq);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage][warp]);
    if (flags & 1) break;
    if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
  }
  if (cur >= 0) flush(a, sm, ws, a.part + ((size_t)cta + cur) * G * PART_STRIDE);
}

template <int G>
__global__ void __launch_bounds__(THREADS, G <= 4 ? 3 : 2) attn_kernel(Args a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<G> &sm = *reinterpret_cast<Smem<G> *>(smem_raw);
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x < a.n_bf) bf16_role<G>(a, sm);
  else hist_role<G>(a, sm, (int)blockIdx.x - a.n_bf);
}

// ---------------------------------------------------------------------------------------------
// Merge: grid (G, Hkv, B), 512 threads; one CTA per (query head of the group, KV head, sequence).
// The history partials of a segment sit in consecutive slots (CTA index + segment index).  Latency
// bound, so the global reads are issued in few dependent rounds: the pool counters (to locate the
// segment's partials), then every partial's (m, l) together with up to OV output values per thread and
// the R_v rows of the un-rotation; the softmax weights are applied once the maximum is known.  The
// un-rotation o[c] = sum_j o_rot[j] R_v[c][j] gives each warp 8 outputs c, its lanes splitting j, so
// that each R_v row is read as one contiguous 512-byte run.
constexpr int MT = 512;
constexpr int MAXPARTS = 1040;
template <int G>
__global__ void __launch_bounds__(MT) merge_kernel(PoolArgs p, const float *part, int n_hist, float *out) {
  constexpr int OV = 36;  // partials per slice issued at once (4 slices: 144 partials)
  __shared__ float wgt[MAXPARTS], lsum[MAXPARTS];
  __shared__ float red[MT / 32];
  __shared__ float Osl[4][D], Obs[4][D], Orot[D];
  __shared__ long long s_pref, s_total;
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z, seg = b * p.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = tid & (D - 1), sl = tid >> 7;
  if (warp == 0) {
    long long total;
    int bb, kk, ll;
    locate(p, 0, bb, kk, ll, total);
    long long run = 0;
    for (int base = 0; base < b; base += 32) {
      const int x = base + lane;
      long long v = (x < b) ? (long long)npages_of(p, x) * p.Hkv : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
      run += v;
    }
    if (lane == 0) { s_pref = run; s_total = total; }
  }
  __syncthreads();
  const int np = npages_of(p, b);
  int nh = 0, i0 = 0;
  if (np > 0) {
    const long long chunk = (s_total + n_hist - 1) / n_hist;
    const long long start = s_pref + (long long)kvh * np, end = start + np;
    i0 = (int)(start / chunk);
    nh = (int)((end - 1) / chunk) - i0 + 1;
  }
  const int nparts = nh + 5;
  const size_t stride = (size_t)G * PART_STRIDE;
  const float *hp = part + ((size_t)i0 + seg) * stride + (size_t)h * PART_STRIDE;
  const float *bp = part + ((size_t)n_hist + (size_t)p.B * p.Hkv + (size_t)seg * 5) * stride + (size_t)h * PART_STRIDE;
  auto slot = [&](int i) { return i < nh ? hp + (size_t)i * stride : bp + (size_t)(i - nh) * stride; };
  float mx = -INFINITY;
  for (int i = tid; i < nparts; i += MT) {
    const float *q = slot(i);
    const float m = q[D];
    wgt[i] = m;
    lsum[i] = q[D + 1];
    mx = fmaxf(mx, m);
  }
  float ov[OV];
#pragma unroll
  for (int k = 0; k < OV; ++k) {
    const int i = sl + 4 * k;
    ov[k] = i < nparts ? slot(i)[ch] : 0.f;
  }
  // R_v rows c = warp + 16 k (k < 8), lane's four columns 4 lane .. 4 lane + 3
  constexpr int UW = MT / 32, UPW = D / UW;
  float4 rv[UPW];
#pragma unroll
  for (int k = 0; k < UPW; ++k)
    rv[k] = reinterpret_cast<const float4 *>(p.R_v + ((size_t)kvh * D + warp + UW * k) * D)[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < MT / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float ls = 0.f;
  for (int i = tid; i < nparts; i += MT) {
    const float e = (wgt[i] == -INFINITY) ? 0.f : exp2f(wgt[i] - M);
    wgt[i] = e;
    ls += e * lsum[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(FULL, ls, o);
  if (lane == 0) red[warp] = ls;
  __syncthreads();
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < MT / 32; ++w) L += red[w];
  // weighted sums: history partials (rotated space) and BF16 partials (original space) apart
  float acc = 0.f, accb = 0.f;
#pragma unroll
  for (int k = 0; k < OV; ++k) {
    const int i = sl + 4 * k;
    const float w = i < nparts ? wgt[i] : 0.f;
    if (i < nh) acc = fmaf(w, ov[k], acc);
    else accb = fmaf(w, ov[k], accb);
  }
  for (int i = sl + 4 * OV; i < nparts; i += 4) {
    if (i < nh) acc = fmaf(wgt[i], slot(i)[ch], acc);
    else accb = fmaf(wgt[i], slot(i)[ch], accb);
  }
  Osl[sl][ch] = acc;
  Obs[sl][ch] = accb;
  __syncthreads();
  if (sl == 0) Orot[ch] = ((Osl[0][ch] + Osl[1][ch]) + Osl[2][ch]) + Osl[3][ch];
  __syncthreads();
  {
    const float4 o4 = reinterpret_cast<const float4 *>(Orot)[lane];
#pragma unroll
    for (int k = 0; k < UPW; ++k) {
      float u = fmaf(rv[k].x, o4.x, fmaf(rv[k].y, o4.y, fmaf(rv[k].z, o4.z, rv[k].w * o4.w)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(FULL, u, o);
      if (lane == 0) Osl[0][warp + UW * k] = u;  // slot 0 of Osl is free again
    }
  }
  __syncthreads();
  if (sl == 0) {
    const float o = Osl[0][ch] + (((Obs[0][ch] + Obs[1][ch]) + Obs[2][ch]) + Obs[3][ch]);
    out[((size_t)b * p.Hq + kvh * G + h) * D + ch] = L > 0.f ? o / L : 0.f;
  }
}

}  // namespace v1

// ---------------------------------------------------------------------------------------------
// Grid of the attention kernel: BF16 CTAs (5 per sequence and KV head) first, then history CTAs
// sized so that both fit in one wave of resident CTAs (history CTAs get at least 3/4 of it).
template <int G>
static int resident_ctas() {
  static int cached = 0;
  if (cached == 0) {
    int dev = 0, sms = 148, occ = 1;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = (int)sizeof(v1::Smem<G>);
    cudaFuncSetAttribute(v1::attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v1::attn_kernel<G>, v1::THREADS, smem) != cudaSuccess ||
        occ < 1)
      occ = 1;
    cached = sms * occ;
  }
  return cached;
}

static int resident_ctas_for(int G) {
  switch (G) {
    case 1: return resident_ctas<1>();
    case 2: return resident_ctas<2>();
    case 4: return resident_ctas<4>();
    default: return resident_ctas<8>();
  }
}

int v1_hist_ctas(const PoolArgs &p) {
  const int slots = resident_ctas_for(p.Hq / p.Hkv);
  const long long nbf = (long long)p.B * p.Hkv * 5;
  long long n = slots - (nbf < slots / 4 ? nbf : slots / 4);
  if (n > 1000) n = 1000;  // the merge kernel gathers at most MAXPARTS partials per segment
  const long long cap = (long long)p.B * p.Hkv * p.max_pages;
  if (cap < n) n = cap;
  return (int)(n < 1 ? 1 : n);
}

size_t v1_ws_bytes(const PoolArgs &p) {
  const int G = p.Hq / p.Hkv;
  const size_t slots = (size_t)v1_hist_ctas(p) + (size_t)p.B * p.Hkv * 6;
  return (size_t)p.B * p.Hq * D * sizeof(float) + slots * G * PART_STRIDE * sizeof(float);
}

// k_new != NULL: the step form (append + demote + query rotation fused in the demote kernel);
// otherwise the query rotation runs as its own kernel.
template <int G>
static cudaError_t launch_v1_g(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                               cudaStream_t s, const uint16_t *k_new = nullptr, const uint16_t *v_new = nullptr) {
  v1::Args a;
  a.p = p;
  a.q = q;
  a.qrot = ws;
  a.part = ws + (size_t)p.B * p.Hq * D;
  a.sm_log2 = sm_scale * 1.4426950408889634f;
  a.n_hist = v1_hist_ctas(p);
  const int nbf = p.B * p.Hkv * 5;
  a.n_bf = nbf;
  const int smem = (int)sizeof(v1::Smem<G>);
  cudaError_t e = cudaFuncSetAttribute(v1::attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (k_new != nullptr) {
    if ((e = launch_demote(p, nullptr, 2, k_new, v_new, s, q, ws)) != cudaSuccess) return e;
  } else if ((e = launch_pdl(v1::qrot_kernel<G>, dim3(p.B * p.Hkv), dim3(512), 0, s, p, q, ws)) != cudaSuccess) {
    return e;
  }
  profile_begin(OSCAR_PROFILE_HISTORY, s);
  if ((e = launch_pdl(v1::attn_kernel<G>, dim3(a.n_hist + nbf), dim3(v1::THREADS), smem, s, a)) != cudaSuccess) return e;
  profile_end(OSCAR_PROFILE_HISTORY, s);
  return launch_pdl(v1::merge_kernel<G>, dim3(G, p.Hkv, p.B), dim3(v1::MT), 0, s, p, (const float *)a.part, a.n_hist,
                    out);
}

cudaError_t launch_decode_v1(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, float *ws,
                             cudaStream_t s) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_v1_g<1>(p, q, out, sm_scale, ws, s);
    case 2: return launch_v1_g<2>(p, q, out, sm_scale, ws, s);
    case 4: return launch_v1_g<4>(p, q, out, sm_scale, ws, s);
    case 8: return launch_v1_g<8>(p, q, out, sm_scale, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_step_v1(const PoolArgs &p, const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q,
                           float *out, float sm_scale, float *ws, cudaStream_t s) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_v1_g<1>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 2: return launch_v1_g<2>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 4: return launch_v1_g<4>(p, q, out, sm_scale, ws, s, k_new, v_new);
    case 8: return launch_v1_g<8>(p, q, out, sm_scale, ws, s, k_new, v_new);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oscar

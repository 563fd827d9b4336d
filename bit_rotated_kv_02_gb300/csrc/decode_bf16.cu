// BF16 paged KV cache: append, bulk prefill and decode attention — the baseline that INT2 decoding
// is compared against.
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "评估结果" (Fig. 5), and "OSCAR:
// Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract: batch-1
// decoding at 100k context is up to about 3x faster with the INT2 history than with a BF16 history,
// because fewer KV bytes are read per decoded token.  These kernels keep every token in BF16 in
// 64-token pages (the layout a paged serving engine uses) so that both sides of that comparison run
// on the same GPU.
//
// Decode: two launches.
//   attn_kernel   the flattened (sequence, KV head, page) space is cut into equal contiguous ranges over
//                 one wave of resident CTAs.  A producer warp streams one page (16 KB of K, 16 KB of
//                 V) per ring stage with four tiled TMA copies of 64 rows x 64 channels (128-byte
//                 swizzle, so that the ldmatrix reads below are free of bank conflicts); four consumer warps take 16
//                 tokens of every page each: S = K q on warp MMAs (m16n8k16, bf16 in, f32
//                 accumulate; tokens on M, query heads of the group on N), a lazily rescaled online
//                 softmax in base 2, and O^T += V^T P on warp MMAs (channels on M, heads on N), with
//                 P split into bf16 hi + lo terms (16 significant bits).  One (m, l, o) partial per
//                 query head is written per (CTA, segment).
//   merge_kernel  LSE-combines the partials of each (sequence, KV head) and normalises.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "oscar_internal.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {

namespace bf {

constexpr int NSTAGE = 6;
constexpr int CONSUMER_WARPS = 4, THREADS = 160;
constexpr int HALF_BYTES = PAGE * D * 2;    // one page of K (or of V) of one KV head: 16 KB
constexpr int STAGE_BYTES = 2 * HALF_BYTES;  // K | V
constexpr float LAZY = 8.f;                  // rescale the running output only when the max grows by > 2^8

struct Args {
  CacheArgs c;
  const uint16_t *q;  // [B][Hq][D] bf16
  float sm_log2;      // softmax_scale * log2(e)
  int n_ctas;
  float *part;        // partial slots [n_ctas + B * Hkv][G][PART_STRIDE]
};

__device__ __forceinline__ int clamp_len(const CacheArgs &c, int b) {
  return max(0, min(c.seq_len[b], c.max_pages * PAGE));
}

// This CTA's share of the flattened (sequence, KV head, page) space: pages [lo, lo + n) with
// chunk = ceil(total / n_ctas), lo = cta * chunk, and the position (b0, kvh0, local0) of page lo with
// the page count np0 and length len0 of sequence b0.  Run by one full warp; results in every lane.
__device__ void locate_range(const CacheArgs &c, int n_ctas, int cta, long long &n, int &b0, int &kvh0,
                             int &local0, int &np0, int &len0) {
  const int lane = threadIdx.x & 31;
  long long total = 0;
  for (int base = 0; base < c.B; base += 32) {
    const int b = base + lane;
    long long v = b < c.B ? (long long)((clamp_len(c, b) + PAGE - 1) / PAGE) * c.Hkv : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    total += v;
  }
  const long long chunk = (total + n_ctas - 1) / n_ctas;
  const long long lo = (long long)cta * chunk;
  n = max(0ll, min(total, lo + chunk) - lo);
  b0 = 0; kvh0 = 0; local0 = 0; np0 = 0; len0 = 0;
  if (n <= 0) return;
  long long run = 0;
  for (int base = 0; base < c.B; base += 32) {
    const int b = base + lane;
    const int len = b < c.B ? clamp_len(c, b) : 0;
    const int np = (len + PAGE - 1) / PAGE;
    const long long v = (long long)np * c.Hkv;
    long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += t;
    }
    const long long excl = run + inc - v;
    const unsigned hit = __ballot_sync(FULL, v > 0 && lo >= excl && lo < excl + v);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const long long e = __shfl_sync(FULL, excl, src);
      np0 = __shfl_sync(FULL, np, src);
      len0 = __shfl_sync(FULL, len, src);
      b0 = base + src;
      kvh0 = (int)((lo - e) / np0);
      local0 = (int)((lo - e) % np0);
      return;
    }
    run += __shfl_sync(FULL, inc, 31);
  }
}

template <int G>
struct Smem {
  uint8_t ring[NSTAGE][STAGE_BYTES];  // 1024-byte aligned (the 128-byte swizzle repeats every 1024 bytes)
  uint64_t full[NSTAGE], empty[NSTAGE], csync;
  int meta_seg[NSTAGE], meta_ntok[NSTAGE], meta_flags[NSTAGE];  // flags: 1 last, 2 abort
  float wm[CONSUMER_WARPS][8], wl[CONSUMER_WARPS][8];
  float wo[CONSUMER_WARPS][G][D];
  long long range_n;
  int b0, kvh0, local0, np0, len0;
};
template <int G>
constexpr int smem_bytes() { return (int)sizeof(Smem<G>) + 1024; }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D += A(16x16, row) * B(16x8, col), bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}
// (lo, hi) -> bf16x2, round to nearest even; low half = lo.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Byte offset of the 16-byte chunk holding channels 8c .. 8c+7 of token row r in a page image written
// as two TMA boxes of {64 channels, 64 rows} (channels 0-63, then 64-127; 8 KB each) with the 128-byte
// swizzle: row r of a box is the 128-byte line r, whose chunk index is XORed with r mod 8.  Eight
// consecutive rows at one chunk index then fall on eight different bank groups.
__device__ __forceinline__ uint32_t chunk_off(int r, int c) {
  return (uint32_t)((c >> 3) * (HALF_BYTES / 2) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct WarpState {
  float m2[2], l[2];  // heads 2t, 2t+1 of this lane's column pair
  float O[8][4];      // O^T tiles: channels 16 mt + g (+8), heads 2t, 2t+1
};

__device__ __forceinline__ void reset(WarpState &ws) {
  ws.m2[0] = ws.m2[1] = -INFINITY;
  ws.l[0] = ws.l[1] = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) ws.O[mt][r] = 0.f;
}

// Bounded barrier among the consumer warps (see the INT2 kernel): an mbarrier with one arrival per
// warp, waited with a time limit that sets the timeout bit.
template <int G>
__device__ __forceinline__ void consumer_sync(Smem<G> &sm, uint32_t &par, uint32_t *err) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.csync);
  const bool ok = __all_sync(FULL, mbar_wait_bounded(&sm.csync, par));
  par ^= 1u;
  if (!ok && (threadIdx.x & 31) == 0) atomicOr(err, OSCAR_DEVERR_TIMEOUT);
}

// B fragments of q for S = K q: k = channel (16 kk + 2t, +1 | +8, +9), n = query head g of the group
// (zero for g >= G).  Read straight from global memory as bf16 pairs.
template <int G>
__device__ __forceinline__ void load_q(const Args &a, int b, int kvh, uint32_t (&bq)[8][2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint32_t *qw = reinterpret_cast<const uint32_t *>(a.q + ((size_t)b * a.c.Hq + kvh * G + min(g, G - 1)) * D);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    bq[kk][0] = g < G ? qw[8 * kk + t] : 0u;
    bq[kk][1] = g < G ? qw[8 * kk + t + 4] : 0u;
  }
}

// Combine the consumer warps' state for one segment into partial slot `slot` (m in log2 units).
template <int G>
__device__ __forceinline__ void flush(const Args &a, Smem<G> &sm, WarpState &ws, uint32_t &par, float *slot) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float l = ws.l[j];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(FULL, l, o);
    const int h = 2 * t + j;
    if (g == 0) { sm.wm[warp][h] = ws.m2[j]; sm.wl[warp][h] = l; }
    if (h < G) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        sm.wo[warp][h][16 * mt + g] = ws.O[mt][j];
        sm.wo[warp][h][16 * mt + g + 8] = ws.O[mt][2 + j];
      }
    }
  }
  consumer_sync(sm, par, a.c.err);
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
  consumer_sync(sm, par, a.c.err);
  reset(ws);
}

// This warp's 16 tokens (rows 16 warp .. 16 warp + 15) of one page; ntok = valid rows of the page.
// Rows past ntok hold whatever the page held: their scores are replaced by -inf, and their value
// rows are zeroed in shared memory first (a zero weight times a non-finite value would still poison
// the sum).
__device__ __forceinline__ void page_pass(uint8_t *kpage, int ntok, float sm_log2, WarpState &ws,
                                          const uint32_t (&bq)[8][2]) {
  const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5), g = lane >> 2;
  const int r0 = 16 * warp;
  uint8_t *vpage = kpage + HALF_BYTES;
  if (ntok < r0 + 16) {
    for (int i = lane; i < 16 * 16; i += 32) {  // row r0 + i / 16, chunk i % 16 (any order: whole rows)
      const int r = r0 + (i >> 4);
      if (r >= ntok) *reinterpret_cast<uint4 *>(vpage + chunk_off(r, i & 15)) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();  // these generic writes precede the next TMA fill of the slot
    __syncwarp();
  }
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t kbase = smem_u32(kpage), vbase = smem_u32(vpage);
  // ---- S = K q: tokens r0 .. r0+15 on M, heads on N; two accumulator chains over the 8 k-steps ----
  float S[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const int r = r0 + ((mi & 1) << 3) + ri;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t A[4];
      ldsm_x4(kbase + chunk_off(r, 2 * kk + (mi >> 1)), A);
      mma_bf16(S[kk & 1], A, bq[kk][0], bq[kk][1]);
    }
  }
  // ---- online softmax (base 2) for heads 2t (c0, c2) and 2t+1 (c1, c3); rows g and g+8 ----
  const bool v0 = r0 + g < ntok, v1 = r0 + g + 8 < ntok;
  float s[4];
  s[0] = v0 ? (S[0][0] + S[1][0]) * sm_log2 : -INFINITY;
  s[1] = v0 ? (S[0][1] + S[1][1]) * sm_log2 : -INFINITY;
  s[2] = v1 ? (S[0][2] + S[1][2]) * sm_log2 : -INFINITY;
  s[3] = v1 ? (S[0][3] + S[1][3]) * sm_log2 : -INFINITY;
  float p[4];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float mx = fmaxf(s[j], s[2 + j]);
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
    if (mx > ws.m2[j] + LAZY) {
      const float alpha = ws.m2[j] == -INFINITY ? 0.f : fast_exp2(ws.m2[j] - mx);
      ws.l[j] *= alpha;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) { ws.O[mt][j] *= alpha; ws.O[mt][2 + j] *= alpha; }
      ws.m2[j] = mx;
    }
    p[j] = fast_exp2(s[j] - ws.m2[j]);
    p[2 + j] = fast_exp2(s[2 + j] - ws.m2[j]);
    ws.l[j] += p[j] + p[2 + j];
  }
  // weights in the accumulator layout (row = token, column pair = heads 2t, 2t+1), split hi + lo,
  // transposed into the B operand of O^T += V^T P (k = token, n = head)
  const uint32_t h0 = pack_bf16x2(p[0], p[1]), h1 = pack_bf16x2(p[2], p[3]);
  const uint32_t l0 = pack_bf16x2(p[0] - bf16_lo(h0), p[1] - bf16_hi(h0));
  const uint32_t l1 = pack_bf16x2(p[2] - bf16_lo(h1), p[3] - bf16_hi(h1));
  const uint32_t bh0 = movmatrix_trans(h0), bh1 = movmatrix_trans(h1);
  const uint32_t bl0 = movmatrix_trans(l0), bl1 = movmatrix_trans(l1);
  // ---- O^T += V^T P: channels 16 mt .. 16 mt + 15 on M (ldmatrix.trans of the token-major rows) ----
  const int rv = r0 + ((mi >> 1) << 3) + ri;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t A[4];
    ldsm_x4_trans(vbase + chunk_off(rv, 2 * mt + (mi & 1)), A);
    mma_bf16(ws.O[mt], A, bh0, bh1);
    mma_bf16(ws.O[mt], A, bl0, bl1);
  }
}

template <int G>
__global__ void __launch_bounds__(THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, Args a) {
  extern __shared__ uint8_t smem_raw[];
  Smem<G> &sm = *reinterpret_cast<Smem<G> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const CacheArgs &c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, cta = blockIdx.x;
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], CONSUMER_WARPS); }
    mbar_init(&sm.csync, CONSUMER_WARPS);
    mbar_fence_init();
  }
  pdl_wait();
  pdl_trigger();
  if (warp == CONSUMER_WARPS) {
    long long n;
    int b0, kvh0, local0, np0, len0;
    locate_range(c, a.n_ctas, cta, n, b0, kvh0, local0, np0, len0);
    if (lane == 0) { sm.range_n = n; sm.b0 = b0; sm.kvh0 = kvh0; sm.local0 = local0; sm.np0 = np0; sm.len0 = len0; }
  }
  __syncthreads();
  const long long n = sm.range_n;
  if (n <= 0) return;

  if (warp == CONSUMER_WARPS) {
    // ---------------- producer warp: one page per stage ----------------
    // The lanes hold a window of 32 page-table entries of the current sequence, refilled in one round
    // trip when the window is used up, so that no page waits on its own page-table read.
    int b = sm.b0, kvh = sm.kvh0, local = sm.local0, np = sm.np0, len = sm.len0;
    int win_b = -1, win_base = 0, pt_reg = -1;
    int stage = 0, it = 0;
    uint32_t phase = 0;
    long long done = 0;
    while (done < n) {
      if (b != win_b || local < win_base || local >= win_base + 32) {
        win_b = b;
        win_base = local;
        const int lp = local + lane;
        pt_reg = lp < np ? c.page_table[(size_t)b * c.max_pages + lp] : -1;
      }
      const int pp = __shfl_sync(FULL, pt_reg, local - win_base);
      bool abort = false;
      if (it >= NSTAGE) {  // the slot is released by all four consumer warps
        const bool okw = lane == 0 ? mbar_wait_bounded(&sm.empty[stage], phase ^ 1) : true;
        abort = !__shfl_sync(FULL, okw, 0);
      }
      if (lane == 0) {
        const bool bad = pp < 0 || pp >= c.num_pages;
        if (abort) atomicOr(c.err, OSCAR_DEVERR_TIMEOUT);
        else if (bad) atomicOr(c.err, OSCAR_DEVERR_PAGE_INDEX);
        sm.meta_seg[stage] = b * c.Hkv + kvh;
        sm.meta_ntok[stage] = (bad || abort) ? 0 : min(PAGE, len - local * PAGE);
        sm.meta_flags[stage] = (done + 1 >= n ? 1 : 0) | (abort ? 2 : 0);
        if (!bad && !abort) {
          uint64_t *bar = &sm.full[stage];
          mbar_arrive_expect_tx(bar, (uint32_t)STAGE_BYTES);
          const int row = (pp * c.Hkv + kvh) * PAGE;  // < 2^31: checked on the host
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d(sm.ring[stage] + hf * (HALF_BYTES / 2), &kmap, 0, hf, row, bar);
            tma_load_3d(sm.ring[stage] + HALF_BYTES + hf * (HALF_BYTES / 2), &vmap, 0, hf, row, bar);
          }
        } else {
          mbar_arrive(&sm.full[stage]);
        }
        if (abort)  // wait (bounded) for copies still in flight into slots the consumers may not read
          for (int k = max(0, it - NSTAGE + 1); k < it; ++k)
            mbar_wait_bounded(&sm.full[k % NSTAGE], (uint32_t)((k / NSTAGE) & 1));
      }
      if (abort) break;
      ++done;
      if (++local == np && done < n) {
        local = 0;
        if (++kvh == c.Hkv) {
          kvh = 0;
          do {
            ++b;
            len = b < c.B ? clamp_len(c, b) : 0;
          } while (b < c.B && len == 0);
          np = (len + PAGE - 1) / PAGE;
        }
      }
      ++it;
      if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
    }
    return;
  }
  // ---------------- consumers ----------------
  WarpState ws;
  reset(ws);
  uint32_t bq[8][2];
  uint32_t par = 0;
  int cur = sm.b0 * c.Hkv + sm.kvh0, stage = 0;
  load_q<G>(a, sm.b0, sm.kvh0, bq);  // overlaps the first page copies
  uint32_t phase = 0;
  while (true) {
    if (!mbar_wait_bounded(&sm.full[stage], phase)) {
      if (lane == 0) atomicOr(c.err, OSCAR_DEVERR_TIMEOUT);
      break;
    }
    const int flags = sm.meta_flags[stage];
    if (flags & 2) break;  // producer aborted
    const int seg = sm.meta_seg[stage];
    if (seg != cur) {
      flush<G>(a, sm, ws, par, a.part + ((size_t)cta + cur) * G * PART_STRIDE);
      cur = seg;
      load_q<G>(a, seg / c.Hkv, seg % c.Hkv, bq);
    }
    const int ntok = sm.meta_ntok[stage];
    if (ntok > 16 * warp) page_pass(sm.ring[stage], ntok, a.sm_log2, ws, bq);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);
    if (flags & 1) break;
    if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
  }
  flush<G>(a, sm, ws, par, a.part + ((size_t)cta + cur) * G * PART_STRIDE);
}

// ---------------------------------------------------------------------------------------------
// Merge: grid (G, Hkv, B), 256 threads (two slices of 128 channels); one CTA per (query head of the
// group, KV head, sequence).  The partials of a segment sit in consecutive slots (CTA index + segment
// index); every partial's (m, l) and up to OV output values per thread are loaded at once.
constexpr int MT = 256, SL = MT / D, OV = 24;
constexpr int MAXPARTS = 1040;
template <int G>
__global__ void __launch_bounds__(MT) merge_kernel(CacheArgs c, const float *part, int n_ctas, float *out) {
  __shared__ float wgt[MAXPARTS], lsum[MAXPARTS];
  __shared__ float red[MT / 32];
  __shared__ float Osl[SL][D];
  __shared__ long long s_pref, s_total;
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z, seg = b * c.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, ch = tid & (D - 1), sl = tid >> 7;
  if (warp == 0) {
    long long total = 0, pref = 0;
    for (int base = 0; base < c.B; base += 32) {
      const int x = base + lane;
      long long v = x < c.B ? (long long)((clamp_len(c, x) + PAGE - 1) / PAGE) * c.Hkv : 0;
      long long u = x < b ? v : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        v += __shfl_xor_sync(FULL, v, o);
        u += __shfl_xor_sync(FULL, u, o);
      }
      total += v;
      pref += u;
    }
    if (lane == 0) { s_pref = pref; s_total = total; }
  }
  __syncthreads();
  const int np = (clamp_len(c, b) + PAGE - 1) / PAGE;
  float *dst = out + ((size_t)b * c.Hq + kvh * G + h) * D;
  if (np == 0) {  // an empty sequence attends to nothing
    if (sl == 0) dst[ch] = 0.f;
    return;
  }
  const long long chunk = (s_total + n_ctas - 1) / n_ctas;
  const long long start = s_pref + (long long)kvh * np, end = start + np;
  const int i0 = (int)(start / chunk);
  const int nparts = min((int)((end - 1) / chunk) - i0 + 1, MAXPARTS);
  const size_t stride = (size_t)G * PART_STRIDE;
  const float *hp = part + ((size_t)i0 + seg) * stride + (size_t)h * PART_STRIDE;
  float mx = -INFINITY;
  for (int i = tid; i < nparts; i += MT) {
    const float m = hp[(size_t)i * stride + D];
    wgt[i] = m;
    lsum[i] = hp[(size_t)i * stride + D + 1];
    mx = fmaxf(mx, m);
  }
  float ov[OV];
#pragma unroll
  for (int k = 0; k < OV; ++k) {
    const int i = sl + SL * k;
    ov[k] = i < nparts ? hp[(size_t)i * stride + ch] : 0.f;
  }
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
    const float e = wgt[i] == -INFINITY ? 0.f : exp2f(wgt[i] - M);
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
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < OV; ++k) {
    const int i = sl + SL * k;
    if (i < nparts) acc = fmaf(wgt[i], ov[k], acc);
  }
  for (int i = sl + SL * OV; i < nparts; i += SL) acc = fmaf(wgt[i], hp[(size_t)i * stride + ch], acc);
  Osl[sl][ch] = acc;
  __syncthreads();
  if (sl == 0) dst[ch] = L > 0.f ? (Osl[0][ch] + Osl[1][ch]) / L : 0.f;
}

// ---------------------------------------------------------------------------------------------
// Append: grid B, 256 threads; token seq_len[b] of every KV head goes to page
// page_table[b][seq_len / 64], row seq_len % 64, then seq_len[b] += 1.
__global__ void __launch_bounds__(256) append_kernel(CacheArgs c, const uint16_t *k_new, const uint16_t *v_new) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int pos = c.seq_len[b];
  bool ok = pos >= 0 && pos < c.max_pages * PAGE;
  int pp = -1;
  if (ok) {
    pp = c.page_table[(size_t)b * c.max_pages + pos / PAGE];
    ok = pp >= 0 && pp < c.num_pages;
    if (!ok && tid == 0) atomicOr(c.err, OSCAR_DEVERR_PAGE_INDEX);
  } else if (tid == 0) {
    atomicOr(c.err, pos < 0 ? OSCAR_DEVERR_COUNTERS : OSCAR_DEVERR_HISTORY_FULL);
  }
  if (!ok) return;
  const int chunks = c.Hkv * 2 * (D / 8);
  for (int i = tid; i < chunks; i += blockDim.x) {
    const int kvh = i / (2 * (D / 8)), kv = (i / (D / 8)) & 1, j = i % (D / 8);
    const uint16_t *src = (kv ? v_new : k_new) + ((size_t)b * c.Hkv + kvh) * D;
    uint16_t *dst = (kv ? c.v_pages : c.k_pages) + (((size_t)pp * c.Hkv + kvh) * PAGE + pos % PAGE) * D;
    reinterpret_cast<uint4 *>(dst)[j] = reinterpret_cast<const uint4 *>(src)[j];
  }
  __syncthreads();
  if (tid == 0) c.seq_len[b] = pos + 1;
}

// Bulk prefill of one sequence: grid (pages, Hkv), 256 threads; tokens [64 p, 64 p + 64) of KV head h of
// k, v (bf16 [len][Hkv][D]) go to page page_table[seq][p].  Block (0, 0) sets seq_len[seq] = len.
__global__ void __launch_bounds__(256) prefill_kernel(CacheArgs c, int seq, int len, const uint16_t *k,
                                                     const uint16_t *v) {
  const int p = blockIdx.x, kvh = blockIdx.y, tid = threadIdx.x;
  const int pp = c.page_table[(size_t)seq * c.max_pages + p];
  if (pp < 0 || pp >= c.num_pages) {
    if (tid == 0) atomicOr(c.err, OSCAR_DEVERR_PAGE_INDEX);
    return;
  }
  const int rows = min(PAGE, len - p * PAGE);
  for (int i = tid; i < 2 * rows * (D / 8); i += blockDim.x) {
    const int kv = i / (rows * (D / 8)), r = (i / (D / 8)) % rows, j = i % (D / 8);
    const uint16_t *src = (kv ? v : k) + ((size_t)(p * PAGE + r) * c.Hkv + kvh) * D;
    uint16_t *dst = (kv ? c.v_pages : c.k_pages) + (((size_t)pp * c.Hkv + kvh) * PAGE + r) * D;
    reinterpret_cast<uint4 *>(dst)[j] = reinterpret_cast<const uint4 *>(src)[j];
  }
  if (p == 0 && kvh == 0 && tid == 0) c.seq_len[seq] = len;
}

}  // namespace bf

// ---------------------------------------------------------------------------------------------
template <int G>
static int bf_resident_ctas() {
  static std::atomic<int> slots[kMaxDevices];
  return per_device(slots, [](int dev) {
    int sms = 148, occ = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(bf::attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, bf::smem_bytes<G>());
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, bf::attn_kernel<G>, bf::THREADS, bf::smem_bytes<G>()) !=
            cudaSuccess ||
        occ < 1)
      occ = 1;
    return sms * occ;
  });
}

int bf16_attn_ctas(const CacheArgs &c) {
  int slots;
  switch (c.Hq / c.Hkv) {
    case 1: slots = bf_resident_ctas<1>(); break;
    case 2: slots = bf_resident_ctas<2>(); break;
    case 4: slots = bf_resident_ctas<4>(); break;
    default: slots = bf_resident_ctas<8>(); break;
  }
  long long n = slots < 1000 ? slots : 1000;  // the merge gathers at most MAXPARTS partials per segment
  const long long cap = (long long)c.B * c.Hkv * c.max_pages;
  if (cap < n) n = cap;
  return (int)(n < 1 ? 1 : n);
}

size_t bf16_ws_bytes(const CacheArgs &c) {
  const int G = c.Hq / c.Hkv;
  const size_t slots = (size_t)bf16_attn_ctas(c) + (size_t)c.B * c.Hkv;
  return slots * G * PART_STRIDE * sizeof(float);
}

// Tensor map over one page array viewed as [rows = num_pages * Hkv * 64][2 halves][64 channels] bf16;
// box = 64 channels of one half x 64 rows (one page of one KV head), 128-byte swizzle.
static cudaError_t page_map(CUtensorMap *map, const uint16_t *base, long long rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) {
    set_last_error("bf16 decode: cuTensorMapEncodeTiled unavailable from the driver");
    return cudaErrorNotSupported;
  }
  cuuint64_t dims[3] = {64, 2, (cuuint64_t)rows};
  cuuint64_t strides[2] = {128, (cuuint64_t)D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)PAGE}, estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("bf16 decode: tensor map rejected (page arrays must be 16-byte aligned)");
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <int G>
static cudaError_t launch_bf16_g(const CacheArgs &c, const uint16_t *q, float *out, float sm_scale, float *ws,
                                 cudaStream_t s, const uint16_t *k_new, const uint16_t *v_new) {
  // The maps depend only on the page arrays; rebuilding them costs host time on every call, so the
  // last pair is kept per thread.
  thread_local CUtensorMap kmap, vmap;
  thread_local const void *kbase = nullptr, *vbase = nullptr;
  thread_local long long mrows = -1;
  const long long rows = (long long)c.num_pages * c.Hkv * PAGE;
  cudaError_t e;
  if (kbase != c.k_pages || vbase != c.v_pages || mrows != rows) {
    kbase = vbase = nullptr;
    if ((e = page_map(&kmap, c.k_pages, rows)) != cudaSuccess) return e;
    if ((e = page_map(&vmap, c.v_pages, rows)) != cudaSuccess) return e;
    kbase = c.k_pages; vbase = c.v_pages; mrows = rows;
  }
  bf::Args a;
  a.c = c;
  a.q = q;
  a.sm_log2 = sm_scale * 1.4426950408889634f;
  a.n_ctas = bf16_attn_ctas(c);
  a.part = ws;
  const int smem = bf::smem_bytes<G>();
  if ((e = cudaFuncSetAttribute(bf::attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  if (k_new != nullptr &&
      (e = launch_pdl(bf::append_kernel, dim3(c.B), dim3(256), 0, s, c, k_new, v_new)) != cudaSuccess)
    return e;
  profile_begin(OSCAR_PROFILE_HISTORY, s);
  if ((e = launch_pdl(bf::attn_kernel<G>, dim3(a.n_ctas), dim3(bf::THREADS), smem, s, kmap, vmap, a)) != cudaSuccess)
    return e;
  profile_end(OSCAR_PROFILE_HISTORY, s);
  return launch_pdl(bf::merge_kernel<G>, dim3(G, c.Hkv, c.B), dim3(bf::MT), 0, s, c, (const float *)ws, a.n_ctas,
                    out);
}

cudaError_t launch_bf16_decode(const CacheArgs &c, const uint16_t *q, float *out, float sm_scale, float *ws,
                               cudaStream_t s, const uint16_t *k_new, const uint16_t *v_new) {
  switch (c.Hq / c.Hkv) {
    case 1: return launch_bf16_g<1>(c, q, out, sm_scale, ws, s, k_new, v_new);
    case 2: return launch_bf16_g<2>(c, q, out, sm_scale, ws, s, k_new, v_new);
    case 4: return launch_bf16_g<4>(c, q, out, sm_scale, ws, s, k_new, v_new);
    case 8: return launch_bf16_g<8>(c, q, out, sm_scale, ws, s, k_new, v_new);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bf16_append(const CacheArgs &c, const uint16_t *k_new, const uint16_t *v_new, cudaStream_t s) {
  return launch_pdl(bf::append_kernel, dim3(c.B), dim3(256), 0, s, c, k_new, v_new);
}

cudaError_t launch_bf16_prefill(const CacheArgs &c, int seq, int len, const uint16_t *k, const uint16_t *v,
                                cudaStream_t s) {
  if (len == 0) return cudaMemsetAsync(c.seq_len + seq, 0, sizeof(int32_t), s);
  bf::prefill_kernel<<<dim3((len + PAGE - 1) / PAGE, c.Hkv), 256, 0, s>>>(c, seq, len, k, v);
  return cudaGetLastError();
}

}  // namespace oscar

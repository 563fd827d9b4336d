// BF16 sink/window partials and the decode step's demotion: the roles shared by the decode kernels.
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": a BF16 kernel handles the
// sink and the recent window of each sequence; the oldest window token is rotated, clipped, quantized,
// packed and demoted into the INT2 history before the step's attention.  Both roles run on the first four
// warps (128 threads) of a CTA; their partials go into the slots the merge kernel reads:
//   BF16 slot of (segment seg, chunk c):   n_hist + B*Hkv + 5*seg + c       (chunk 0 sink, 1..4 window)
//   demoted-token slot of segment seg:     n_hist + 6*B*Hkv + seg
// each G x PART_STRIDE floats (o[128], m (log2 units), l).
#pragma once

#include "oscar_internal.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace part {

constexpr int BF_WARPS = 4;

// The step's pool state after its demotion and append, from the counters before the step; the same
// decisions as the demotion kernel (demote when the window is full and the target page is valid;
// a demotion that cannot be stored blocks the append too).
struct StepState {
  bool ok;        // counters valid
  bool want;      // the window is full: its oldest token is due for demotion
  bool demote;    // the oldest window token moves to history position hist_len
  bool append;    // the new token is stored
  bool to_sink;   // ... into the sink (else into the window)
  int page;       // the page-table entry of history row hl (read when the window is full)
  int slen, hl, rs, rl;        // before
  int nslen, nhl, nrs, nrl;    // after
};
__device__ __forceinline__ StepState step_state(const PoolArgs &p, int b) {
  StepState st;
  st.slen = p.sink_len[b]; st.hl = p.hist_len[b]; st.rs = p.recent_start[b]; st.rl = p.recent_len[b];
  st.ok = st.slen >= 0 && st.slen <= SINK && st.hl >= 0 && st.rs >= 0 && st.rs < RECENT && st.rl >= 0 &&
          st.rl <= RECENT;
  const bool want = st.ok && st.rl == RECENT;
  st.want = want;
  st.demote = false;
  st.page = -1;
  if (want && st.hl / PAGE < p.max_pages) {
    st.page = p.page_table[(size_t)b * p.max_pages + st.hl / PAGE];
    st.demote = st.page >= 0 && st.page < p.num_pages;
  }
  st.append = st.ok && !(want && !st.demote);
  st.nslen = st.slen; st.nhl = st.hl; st.nrs = st.rs; st.nrl = st.rl;
  if (st.demote) { st.nhl = st.hl + 1; st.nrs = (st.rs + 1) % RECENT; st.nrl = st.rl - 1; }
  st.to_sink = st.append && st.nslen < SINK && st.nhl == 0 && st.nrl == 0;
  if (st.append) {
    if (st.to_sink) st.nslen += 1;
    else st.nrl += 1;
  }
  return st;
}


// Shared memory of the BF16 role (the argument struct A carries p, q, sm_log2, n_hist, part, step, k_new,
// v_new); demotion scratch is separate (DEMOTE_SCRATCH bytes).
template <int G>
struct BfSmem {
  alignas(16) float qr[D][G];  // the queries, channel-major (a channel's G values adjacent, read in 8-byte pairs)
  float wm[BF_WARPS][G], wl[BF_WARPS][G];
  float wo[BF_WARPS][G][D];
  float pbuf[BF_WARPS][G][16];
};
constexpr int DEMOTE_SCRATCH = (D + 2 * 4 * 32 * 4) * 4 + D / 4 + 16 + 64 + 16;

// ---------------------------------------------------------------------------------------------
// Decode-step demotion, run by BF16 CTAs before their chunk:
// the sink CTA (chunk 0) demotes the window's oldest K vector, the first window CTA (chunk 1) its V
// vector (slot recent_start, unchanged until the merge).  The vector is rotated, clipped and quantized
// exactly as the demotion kernel does (four warps, 32 rows of R each in two batches of 16; any summation
// order: quantize_from_dots bounds it), its codes, scale and zero are stored into history row hist_len
// (which no consumer of this step reads), and the demoted token becomes one more rotated-space partial of
// every query head of the group: the K CTA writes m = its score q_rot . (zero + scale * level[code]) *
// log2(e) * softmax_scale (a compensated sum) and l = 1, the V CTA o = its dequantized V.  Without a
// demotion the slot holds an empty partial.  The scratch lives in the page ring, which BF16 CTAs do not
// use.
template <int G, class A>
__device__ __noinline__ void demote_role(const A &a, uint8_t *scratch, int b, int kvh, int seg, const StepState &st,
                                         int kv, const float *qrot_rows, bool wait_qrot) {
  const PoolArgs &p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!OSCAR_DCHECK(seg >= 0 && seg < p.B * p.Hkv, p.err)) return;
  float *dslot = a.part + ((size_t)a.n_hist + (size_t)p.B * p.Hkv * 6 + seg) * G * PART_STRIDE;
  if (!st.demote) {
    for (int i = tid; i < G * PART_STRIDE; i += 128) {
      const int c = i % PART_STRIDE;
      if (kv == 0 ? (c == D || c == D + 1) : c < D) dslot[i] = c == D ? -INFINITY : 0.f;
    }
    return;
  }
  float *xs = reinterpret_cast<float *>(scratch);     // [D]: the vector
  float *pacc = xs + D;                                // [4 warps][32 lanes][4]
  float *psab = pacc + 4 * 32 * 4;
  uint8_t *dcode = reinterpret_cast<uint8_t *>(psab + 4 * 32 * 4);  // [D / 4]
  uint16_t *dsz = reinterpret_cast<uint16_t *>(dcode + D / 4);      // scale[4], zero[4] (one per group)
  float *red = reinterpret_cast<float *>(dsz + 8);                  // [16]: the quantizer's group extremes
  const float *Rw = (kv == 0 ? p.R_k : p.R_v) + (size_t)kvh * D * D;
  const float *cb = kv == 0 ? p.cb_k : p.cb_v;
  // this warp's first 16 rows of R are requested with the vector (they do not depend on it)
  float4 rrow[16];
  {
    const float4 *R4 = reinterpret_cast<const float4 *>(Rw) + (size_t)(32 * warp) * (D / 4) + lane;
#pragma unroll
    for (int i = 0; i < 16; ++i) rrow[i] = R4[i * (D / 4)];
  }
  if (warp == 0) {
    const uint2 xw = reinterpret_cast<const uint2 *>((kv == 0 ? p.recent_k : p.recent_v) +
                                                     (((size_t)b * p.Hkv + kvh) * RECENT + st.rs) * D)[lane];
    xs[4 * lane + 0] = bf16_to_f32(xw.x & 0xffffu);
    xs[4 * lane + 1] = bf16_to_f32(xw.x >> 16);
    xs[4 * lane + 2] = bf16_to_f32(xw.y & 0xffffu);
    xs[4 * lane + 3] = bf16_to_f32(xw.y >> 16);
  }
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, sab[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int bt = 0; bt < 2; ++bt) {
    const int r0 = 32 * warp + 16 * bt;
    if (bt == 1) {
      const float4 *R4 = reinterpret_cast<const float4 *>(Rw) + (size_t)r0 * (D / 4) + lane;
#pragma unroll
      for (int i = 0; i < 16; ++i) rrow[i] = R4[i * (D / 4)];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float xi = xs[r0 + i], ax = fabsf(xi);
      acc[0] = fmaf(xi, rrow[i].x, acc[0]);
      acc[1] = fmaf(xi, rrow[i].y, acc[1]);
      acc[2] = fmaf(xi, rrow[i].z, acc[2]);
      acc[3] = fmaf(xi, rrow[i].w, acc[3]);
      sab[0] = fmaf(ax, fabsf(rrow[i].x), sab[0]);
      sab[1] = fmaf(ax, fabsf(rrow[i].y), sab[1]);
      sab[2] = fmaf(ax, fabsf(rrow[i].z), sab[2]);
      sab[3] = fmaf(ax, fabsf(rrow[i].w), sab[3]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) { pacc[(warp * 32 + lane) * 4 + k] = acc[k]; psab[(warp * 32 + lane) * 4 + k] = sab[k]; }
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
  {  // thread e quantizes element e (its four warps' partial sums, added as one warp would)
    const int k = tid & 3, l = tid >> 2;
    const float a = (pacc[l * 4 + k] + pacc[(32 + l) * 4 + k]) + (pacc[(64 + l) * 4 + k] + pacc[(96 + l) * 4 + k]);
    const float sb = (psab[l * 4 + k] + psab[(32 + l) * 4 + k]) + (psab[(64 + l) * 4 + k] + psab[(96 + l) * 4 + k]);
    QuantStats qst{0, 0, 0};
    quantize_from_dots_cta(xs, Rw, Rw, D, a, sb, (kv == 0 ? p.clip_k : p.clip_v)[kvh], p.g, dcode, dsz, dsz + 4, qst,
                           cb != nullptr ? cb + 4 * kvh : nullptr, red, 1);
  }
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
  if (tid < D / 4) {  // the demoted codes, scale and zero into history row hist_len (its page: step_state's)
    const int page = st.page;
    const size_t row = ((size_t)page * p.Hkv + kvh) * PAGE + st.hl % PAGE;
    if (OSCAR_DCHECK(page >= 0 && page < p.num_pages, p.err)) {
    (kv == 0 ? p.codes_k : p.codes_v)[row * (D / 4) + tid] = dcode[tid];
    if (tid < p.ng) {
      (kv == 0 ? p.scale_k : p.scale_v)[row * p.ng + tid] = dsz[tid];
      (kv == 0 ? p.zero_k : p.zero_v)[row * p.ng + tid] = dsz[4 + tid];
    }
    }
  }
  // dequantization levels (the codes themselves without a codebook); group of channel c: c / g
  auto level = [&](uint32_t c) { return cb != nullptr ? cb[4 * kvh + c] : (float)c; };
  if (kv == 1) {  // o: the dequantized rotated V, the same for every head
    for (int i = tid; i < G * D; i += 128) {
      const int c = i % D, gr = c / p.g;
      dslot[(i / D) * PART_STRIDE + c] =
          fmaf(level((dcode[c / 4] >> (2 * (c & 3))) & 3u), bf16_to_f32(dsz[gr]), bf16_to_f32(dsz[4 + gr]));
    }
    return;
  }
  if (wait_qrot) pdl_wait();  // q_rot comes from the previous kernel on the stream: it has completed
  const uint32_t cw = dcode[lane];  // K codes of channels 4 lane .. 4 lane + 3 (all in group 4 lane / g)
  const float sc = bf16_to_f32(dsz[4 * lane / p.g]), zr = bf16_to_f32(dsz[4 + 4 * lane / p.g]);
  for (int h = warp; h < G; h += 4) {
    const float4 q4 = reinterpret_cast<const float4 *>(qrot_rows + (size_t)h * D)[lane];
    const float qr[4] = {q4.x, q4.y, q4.z, q4.w};
    float dc = 0.f, dce = 0.f, sq = 0.f;  // sum of q_rot * level with its rounding errors
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float cf = level((cw >> (2 * k)) & 3u);
      const float pr = qr[k] * cf, pe = fmaf(qr[k], cf, -pr);
      float t, e2;
      two_sum_f32(dc, pr, t, e2);
      dc = t;
      dce += e2 + pe;
      sq += qr[k];
    }
    if (p.ng > 1) {
      // one group per lane: the lane's partial with its group's scale and zero (one rounding), then the
      // compensated sum over the lanes
      dc = fmaf(sc, dc + dce, zr * sq);
      dce = 0.f;
      sq = 0.f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float d2 = __shfl_xor_sync(FULL, dc, o);
      dce += __shfl_xor_sync(FULL, dce, o);
      float t, e2;
      two_sum_f32(dc, d2, t, e2);
      dc = t;
      dce += e2;
      sq += __shfl_xor_sync(FULL, sq, o);
    }
    if (lane == 0) {
      dslot[h * PART_STRIDE + D] = a.sm_log2 * (p.ng > 1 ? dc + dce : fmaf(sc, dc + dce, zr * sq));
      dslot[h * PART_STRIDE + D + 1] = 1.f;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// BF16 sink/recent chunk: block index = segment * 5 + chunk (chunk 0 = sink, 1..4 = recent tokens
// 64(chunk-1) .. 64 chunk - 1 counted from the oldest).
template <int G, class A, class SM, class QR>
__device__ __forceinline__ void bf16_role(const A &a, SM &sm, int idx, uint8_t *scratch, QR qrot_rows) {
  const PoolArgs &p = a.p;
  const int seg = idx / 5, chunk = idx % 5, b = seg / p.Hkv, kvh = seg % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!OSCAR_DCHECK(seg < p.B * p.Hkv, p.err)) return;
  float *slot = a.part + ((size_t)a.n_hist + (size_t)p.B * p.Hkv + (size_t)seg * 5 + chunk) * G * PART_STRIDE;
  if (warp >= BF_WARPS) return;
  // the queries are requested first (they do not depend on the counters)
  constexpr int QPT = (G * D + 127) / 128;
  uint16_t qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int i = tid + 128 * k;
    qv[k] = i < G * D ? a.q[((size_t)b * p.Hq + kvh * G) * D + i] : 0;
  }
  int slen, rs, rl;
  int new_at = -1;  // step form: the chunk-local index of the new token (read from k_new / v_new)
  StepState st{};
  if (a.step) {
    st = step_state(p, b);
    slen = st.nslen; rs = st.nrs; rl = st.nrl;
    if (st.append) {
      if (st.to_sink) new_at = chunk == 0 ? st.slen : -1;
      else if (chunk > 0) new_at = st.nrl - 1 - (chunk - 1) * 64;
    }
  } else {
    slen = p.sink_len[b]; rs = p.recent_start[b]; rl = p.recent_len[b];
  }
  slen = max(0, min(slen, SINK)); rs = max(0, min(rs, RECENT - 1)); rl = max(0, min(rl, RECENT));
  const int n = (chunk == 0) ? slen : max(0, min(64, rl - (chunk - 1) * 64));
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int i = tid + 128 * k;
    if (i < G * D) sm.qr[i % D][i / D] = bf16_to_f32(qv[k]);
  }
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
  // the demotion first: its R rows are read while the history CTAs are still starting, and the CTA's own
  // chunk then ends about when a chunk without a demotion would have
  if (a.step && chunk < 2) {
    bool wait_qrot = false;
    const float *qr = chunk == 0 ? qrot_rows(b, kvh, sm, wait_qrot) : nullptr;
    demote_role<G>(a, scratch, b, kvh, seg, st, chunk, qr, wait_qrot);
  }
  const uint16_t *kb = chunk == 0 ? p.sink_k + ((size_t)b * p.Hkv + kvh) * SINK * D
                                  : p.recent_k + ((size_t)b * p.Hkv + kvh) * RECENT * D;
  const uint16_t *vb = chunk == 0 ? p.sink_v + ((size_t)b * p.Hkv + kvh) * SINK * D
                                  : p.recent_v + ((size_t)b * p.Hkv + kvh) * RECENT * D;
  auto row_of = [&](int i) { return chunk == 0 ? i : (rs + (chunk - 1) * 64 + i) % RECENT; };
  const uint16_t *kn = a.step ? a.k_new + ((size_t)b * p.Hkv + kvh) * D : nullptr;
  const uint16_t *vn = a.step ? a.v_new + ((size_t)b * p.Hkv + kvh) * D : nullptr;
  auto krow = [&](int i) { return i == new_at ? kn : kb + (size_t)row_of(i) * D; };
  auto vrow = [&](int i) { return i == new_at ? vn : vb + (size_t)row_of(i) * D; };
  // QK: lane -> token (lane & 15) of this warp's 16, channel half (lane >> 4)
  const int tk = 16 * warp + (lane & 15), hf = lane >> 4;
  const bool valid = tk < n;
  // the products of two bf16 values are exact in float32; their sum carries its rounding errors
  // (TwoSum), so that the score is the exact dot product rounded about once: logits of several
  // hundred with two tokens sharing the weight need that accuracy
  // (heads in pairs on paired float32 operations, each lane rounding as the scalar TwoSum does)
  float dot[G], cmp[G];
#pragma unroll
  for (int h = 0; h < G; ++h) dot[h] = cmp[h] = 0.f;
  if (valid) {
    const uint4 *kr = reinterpret_cast<const uint4 *>(krow(tk) + hf * 64);
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = kr[i];
    constexpr int GP = G / 2;  // head pairs
    float2 d2[GP > 0 ? GP : 1], c2[GP > 0 ? GP : 1];
#pragma unroll
    for (int k = 0; k < GP; ++k) d2[k] = c2[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float kv = bf16_to_f32((ws[e >> 1] >> (16 * (e & 1))) & 0xffffu);
        const float *qc = sm.qr[hf * 64 + 8 * i + e];
#pragma unroll
        for (int k = 0; k < GP; ++k) {
          const float2 q2 = *reinterpret_cast<const float2 *>(qc + 2 * k);
          const float2 pr = fmul2(make_float2(kv, kv), q2);  // exact: products of two bf16 values
          const float2 s = fadd2(d2[k], pr), bp = fsub2(s, d2[k]);
          const float2 er = fadd2(fsub2(d2[k], fsub2(s, bp)), fsub2(pr, bp));
          d2[k] = s;
          c2[k] = fadd2(c2[k], er);
        }
        if constexpr (G % 2 == 1) {
          const float pr = kv * qc[G - 1];
          float t, e2;
          two_sum_f32(dot[G - 1], pr, t, e2);
          dot[G - 1] = t;
          cmp[G - 1] += e2;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < GP; ++k) {
      dot[2 * k] = d2[k].x; dot[2 * k + 1] = d2[k].y;
      cmp[2 * k] = c2[k].x; cmp[2 * k + 1] = c2[k].y;
    }
  }
  float m2[G], l[G], o[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    {
      const float d2 = __shfl_xor_sync(FULL, dot[h], 16), c2 = __shfl_xor_sync(FULL, cmp[h], 16);
      float t, e2;
      two_sum_f32(dot[h], d2, t, e2);
      dot[h] = t + ((cmp[h] + c2) + e2);
    }
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
    vv[j] = t2 < n ? reinterpret_cast<const uint2 *>(vrow(t2))[lane] : make_uint2(0, 0);
  }
  // (channel pairs on paired float32 FMAs)
  float2 ov[G][2];
#pragma unroll
  for (int h = 0; h < G; ++h) ov[h][0] = ov[h][1] = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 v01 = make_float2(bf16_to_f32(vv[j].x & 0xffffu), bf16_to_f32(vv[j].x >> 16));
    const float2 v23 = make_float2(bf16_to_f32(vv[j].y & 0xffffu), bf16_to_f32(vv[j].y >> 16));
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float pj = sm.pbuf[warp][h][j];
      ov[h][0] = ffma2(make_float2(pj, pj), v01, ov[h][0]);
      ov[h][1] = ffma2(make_float2(pj, pj), v23, ov[h][1]);
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    o[h][0] = ov[h][0].x; o[h][1] = ov[h][0].y;
    o[h][2] = ov[h][1].x; o[h][3] = ov[h][1].y;
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
    for (int w = 0; w < BF_WARPS; ++w) M = fmaxf(M, sm.wm[w][h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < BF_WARPS; ++w) {
        const float e = sm.wm[w][h] == -INFINITY ? 0.f : exp2f(sm.wm[w][h] - M);
        L += e * sm.wl[w][h];
        O += e * sm.wo[w][h][tid];
      }
    }
    slot[h * PART_STRIDE + tid] = O;
    if (tid == 0) { slot[h * PART_STRIDE + D] = M; slot[h * PART_STRIDE + D + 1] = L; }
  }
}


}  // namespace part
}  // namespace oscar

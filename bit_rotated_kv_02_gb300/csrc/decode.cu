// Decode attention over the three-segment pool.
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": at decode the INT2
// kernel unpacks, dequantizes with scale/zero point and accumulates in floating point; a BF16 kernel
// handles sink/recent; an online softmax merge combines the two results.
// "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract:
// a custom INT2 attention kernel compatible with paged KV-cache serving.
//
// Work split: the history of every (sequence, KV head) is cut into `splits` page ranges; each CTA
// streams its pages, scores the G query heads of the group with the rotated query q·R_k, and writes
// one (m, l, o_rot) partial per head.  A second kernel computes the BF16 sink/recent partial.  The
// merge kernel LSE-combines the history partials, un-rotates with R_v^T and merges the BF16 partial.
#include "oscar_internal.cuh"
#include "kernels.h"

namespace oscar {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ float level(uint32_t code, float4 l) {
  return code < 2 ? (code == 0 ? l.x : l.y) : (code == 2 ? l.z : l.w);
}

// true when token j of the chunk has weight 0 for every head (an invalid token: its staged row was not written)
template <int G>
__device__ __forceinline__ bool s_all_zero(float (*pbuf)[32], int j) {
  bool z = true;
#pragma unroll
  for (int h = 0; h < G; ++h) z = z && pbuf[h][j] == 0.f;
  return z;
}

// Online-softmax update of one 32-token chunk for G heads; scores s[h] are lane-local (one token per
// lane), o[h][k] are lane-local output channels 4*lane+k.  p values go to pbuf[h][lane].
template <int G>
__device__ __forceinline__ void softmax_chunk(const float (&s)[G], float (&m)[G], float (&l)[G], float (&o)[G][4],
                                              float (*pbuf)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float mnew = fmaxf(m[h], warp_max(s[h]));
    const float alpha = (m[h] == -INFINITY) ? 0.f : expf(m[h] - mnew);
    const float pr = (s[h] == -INFINITY) ? 0.f : expf(s[h] - mnew);
    l[h] = l[h] * alpha + warp_sum(pr);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[h][k] *= alpha;
    m[h] = mnew;
    pbuf[h][lane] = pr;
  }
  __syncwarp();
}

// Combine the 4 warps' (m, l, o) and store one partial per head: part[h] = {o[0..127], m, l}.
template <int G>
__device__ __forceinline__ void store_partial(const float (&m)[G], const float (&l)[G], const float (&o)[G][4],
                                              float *part) {
  __shared__ float wm[4][G], wl[4][G];
  __shared__ float wo[4][G][D];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) { wm[warp][h] = m[h]; wl[warp][h] = l[h]; }
#pragma unroll
    for (int k = 0; k < 4; ++k) wo[warp][h][4 * lane + k] = o[h][k];
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w][h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float e = (wm[w][h] == -INFINITY) ? 0.f : expf(wm[w][h] - M);
        L += e * wl[w][h];
        O += e * wo[w][h][tid];
      }
    }
    part[h * PART_STRIDE + tid] = O;
    if (tid == 0) { part[h * PART_STRIDE + D] = M; part[h * PART_STRIDE + D + 1] = L; }
  }
}

// ---------------------------------------------------------------------------------------------
// INT2 history partials: grid (splits, Hkv, B), 128 threads.  Token-per-lane scoring; channel
// chunks per lane for the PV accumulation.
template <int G>
__global__ void __launch_bounds__(128) hist_partial_kernel(PoolArgs p, const uint16_t *q, float sm_scale, int splits,
                                                           int pps, float *ws) {
  __shared__ float qs[G][D];
  __shared__ float qr[D][G];
  __shared__ float qsum[G][4];
  __shared__ float pbuf[4][G][32];
  __shared__ uint4 vrow_s[4][32][2];      // per warp: the V codes of the chunk's 32 tokens (32 bytes each)
  __shared__ uint16_t vsz_s[4][32][8];    // per warp: their V scales [0, ng) and zeros [4, 4 + ng)
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = p.g, ng = p.ng;
  for (int i = tid; i < G * D; i += 128)
    qs[i / D][i % D] = bf16_to_f32(q[((size_t)b * p.Hq + kvh * G + i / D) * D + (i % D)]);
  __syncthreads();
  {  // q_rot = q · R_k (row-vector convention); thread tid computes channel tid of every head
    const float *R = p.R_k + (size_t)kvh * D * D;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;
    for (int i = 0; i < D; ++i) {
      const float r = R[i * D + tid];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = fmaf(qs[h][i], r, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) qr[tid][h] = acc[h];
  }
  __syncthreads();
  if (tid < G * ng) {
    const int h = tid / ng, gi = tid % ng;
    float s = 0.f;
    for (int c = gi * g; c < (gi + 1) * g; ++c) s += qr[c][h];
    qsum[h][gi] = s;
  }
  __syncthreads();

  int hl = p.hist_len[b];
  if (hl < 0 || hl > p.max_pages * PAGE) {
    if (tid == 0) atomicOr(p.err, OSCAR_DEVERR_COUNTERS);
    hl = max(0, min(hl, p.max_pages * PAGE));
  }
  const int t0 = split * pps * PAGE;
  const int t1 = min(t0 + pps * PAGE, hl);
  // dequantization levels of this KV head (the uniform 0, 1, 2, 3 without a codebook)
  const float4 lk = p.cb_k != nullptr ? reinterpret_cast<const float4 *>(p.cb_k)[kvh] : make_float4(0.f, 1.f, 2.f, 3.f);
  const float4 lv = p.cb_v != nullptr ? reinterpret_cast<const float4 *>(p.cb_v)[kvh] : make_float4(0.f, 1.f, 2.f, 3.f);
  const int32_t *pt = p.page_table + (size_t)b * p.max_pages;

  float m[G], l[G], o[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY; l[h] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) o[h][k] = 0.f;
  }
  for (int base = t0 + warp * 32; base < t1; base += 128) {
    const int t = base + lane;
    bool valid = t < t1;
    int page = -1;
    if (valid) {
      page = pt[t / PAGE];
      if (page < 0 || page >= p.num_pages) { valid = false; atomicOr(p.err, OSCAR_DEVERR_PAGE_INDEX); }
    }
    float s[G];
    // this lane's token's V row and its scales / zeros, staged for the PV loop (one round of loads)
    if (valid) {
      const size_t row = ((size_t)page * p.Hkv + kvh) * PAGE + (t % PAGE);
      const uint4 *vp = reinterpret_cast<const uint4 *>(p.codes_v + row * (D / 4));
      vrow_s[warp][lane][0] = vp[0];
      vrow_s[warp][lane][1] = vp[1];
      for (int gi = 0; gi < ng; ++gi) {
        vsz_s[warp][lane][gi] = p.scale_v[row * ng + gi];
        vsz_s[warp][lane][4 + gi] = p.zero_v[row * ng + gi];
      }
    }
    if (valid) {
      const size_t row = ((size_t)page * p.Hkv + kvh) * PAGE + (t % PAGE);
      const uint4 *cp = reinterpret_cast<const uint4 *>(p.codes_k + row * (D / 4));
      const uint4 w0 = cp[0], w1 = cp[1];
      const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      float sg[G], r[G];
#pragma unroll
      for (int h = 0; h < G; ++h) { sg[h] = 0.f; r[h] = 0.f; }
#pragma unroll
      for (int w = 0; w < 8; ++w) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float cf = level((words[w] >> (2 * j)) & 3u, lk);
          const int c = 16 * w + j;
#pragma unroll
          for (int h = 0; h < G; ++h) r[h] = fmaf(cf, qr[c][h], r[h]);
        }
        if (((w + 1) * 16) % g == 0) {  // end of a group
          const int gi = (16 * w) / g;
          const float sc = bf16_to_f32(p.scale_k[row * ng + gi]);
          const float z = bf16_to_f32(p.zero_k[row * ng + gi]);
#pragma unroll
          for (int h = 0; h < G; ++h) { sg[h] += sc * r[h] + z * qsum[h][gi]; r[h] = 0.f; }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = sg[h] * sm_scale;
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = -INFINITY;
    }
    softmax_chunk<G>(s, m, l, o, pbuf[warp]);  // ends with a __syncwarp: the staged rows are visible
    const int nv = min(32, t1 - base);
    const int gi = (4 * lane) / g;
    for (int j = 0; j < nv; ++j) {
      if (pbuf[warp][0][j] == 0.f && (G == 1 || s_all_zero<G>(pbuf[warp], j))) continue;  // invalid or no weight
      const uint32_t byte = reinterpret_cast<const uint8_t *>(&vrow_s[warp][j][0])[lane];
      const float sc = bf16_to_f32(vsz_s[warp][j][gi]);
      const float z = bf16_to_f32(vsz_s[warp][j][4 + gi]);
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = fmaf(level((byte >> (2 * k)) & 3u, lv), sc, z);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pj = pbuf[warp][h][j];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[h][k] = fmaf(pj, v[k], o[h][k]);
      }
    }
    __syncwarp();
  }
  float *part = ws + (((size_t)b * p.Hkv + kvh) * (splits + 1) + split) * G * PART_STRIDE;
  store_partial<G>(m, l, o, part);
}

// ---------------------------------------------------------------------------------------------
// BF16 sink + recent partial: grid (Hkv, B), 128 threads.  Written to partial slot `splits`.
template <int G>
__global__ void __launch_bounds__(128) bf16_partial_kernel(PoolArgs p, const uint16_t *q, float sm_scale, int splits,
                                                           float *ws) {
  __shared__ float qs[D][G];
  __shared__ float pbuf[4][G][32];
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < G * D; i += 128)
    qs[i % D][i / D] = bf16_to_f32(q[((size_t)b * p.Hq + kvh * G + i / D) * D + (i % D)]);
  __syncthreads();
  int slen = p.sink_len[b], rs = p.recent_start[b], rl = p.recent_len[b];
  if (slen < 0 || slen > SINK || rs < 0 || rs >= RECENT || rl < 0 || rl > RECENT) {
    if (tid == 0) atomicOr(p.err, OSCAR_DEVERR_COUNTERS);
    slen = max(0, min(slen, SINK)); rs = max(0, min(rs, RECENT - 1)); rl = max(0, min(rl, RECENT));
  }
  const int n = slen + rl;
  const uint16_t *sk = p.sink_k + ((size_t)b * p.Hkv + kvh) * SINK * D;
  const uint16_t *sv = p.sink_v + ((size_t)b * p.Hkv + kvh) * SINK * D;
  const uint16_t *rk = p.recent_k + ((size_t)b * p.Hkv + kvh) * RECENT * D;
  const uint16_t *rv = p.recent_v + ((size_t)b * p.Hkv + kvh) * RECENT * D;
  float m[G], l[G], o[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY; l[h] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) o[h][k] = 0.f;
  }
  for (int base = warp * 32; base < n; base += 128) {
    const int j = base + lane;
    float s[G];
    if (j < n) {
      const uint16_t *krow = j < slen ? sk + (size_t)j * D : rk + (size_t)((rs + j - slen) % RECENT) * D;
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
      const uint4 *k4 = reinterpret_cast<const uint4 *>(krow);
#pragma unroll 4
      for (int c8 = 0; c8 < D / 8; ++c8) {
        const uint4 w = k4[c8];
        const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float kv = bf16_to_f32((ws4[e / 2] >> (16 * (e % 2))) & 0xffffu);
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] = fmaf(kv, qs[8 * c8 + e][h], acc[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = acc[h] * sm_scale;
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = -INFINITY;
    }
    softmax_chunk<G>(s, m, l, o, pbuf[warp]);
    const int nv = min(32, n - base);
    for (int jj = 0; jj < nv; ++jj) {
      const int j2 = base + jj;
      const uint16_t *vrow = j2 < slen ? sv + (size_t)j2 * D : rv + (size_t)((rs + j2 - slen) % RECENT) * D;
      const uint2 w = reinterpret_cast<const uint2 *>(vrow)[lane];
      const float v[4] = {bf16_to_f32(w.x & 0xffffu), bf16_to_f32(w.x >> 16), bf16_to_f32(w.y & 0xffffu),
                          bf16_to_f32(w.y >> 16)};
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pj = pbuf[warp][h][jj];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[h][k] = fmaf(pj, v[k], o[h][k]);
      }
    }
    __syncwarp();
  }
  float *part = ws + (((size_t)b * p.Hkv + kvh) * (splits + 1) + splits) * G * PART_STRIDE;
  store_partial<G>(m, l, o, part);
}

// ---------------------------------------------------------------------------------------------
// Merge: grid (Hkv, B), 128 threads (thread = channel).  LSE-combine the history partials in
// rotated space, un-rotate (o = o_rot · R_v^T, i.e. o[i] = sum_j o_rot[j] R_v[i][j]), then merge
// the BF16 partial and normalise.
template <int G>
__global__ void __launch_bounds__(128) merge_kernel(PoolArgs p, int splits, const float *ws, float *out) {
  extern __shared__ float Rs[];  // [D][D+1]
  __shared__ float orot[D];
  const int kvh = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const float *R = p.R_v + (size_t)kvh * D * D;
  for (int i = tid; i < D * D; i += 128) Rs[(i / D) * (D + 1) + (i % D)] = R[i];
  const float *base = ws + ((size_t)b * p.Hkv + kvh) * (splits + 1) * G * PART_STRIDE;
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, base[(s * G + h) * PART_STRIDE + D]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < splits; ++s) {
        const float *pp = base + (s * G + h) * PART_STRIDE;
        const float ms = pp[D];
        if (ms == -INFINITY) continue;
        const float e = expf(ms - M);
        L += e * pp[D + 1];
        O += e * pp[tid];
      }
    }
    __syncthreads();
    orot[tid] = O;
    __syncthreads();
    float Ou = 0.f;
    for (int j = 0; j < D; ++j) Ou = fmaf(Rs[tid * (D + 1) + j], orot[j], Ou);
    const float *pb = base + (splits * G + h) * PART_STRIDE;
    const float mb = pb[D], lb = pb[D + 1];
    const float mm = fmaxf(M, mb);
    const float wh = (M == -INFINITY) ? 0.f : expf(M - mm);
    const float wb = (mb == -INFINITY) ? 0.f : expf(mb - mm);
    const float den = wh * L + wb * lb;
    out[((size_t)b * p.Hq + kvh * G + h) * D + tid] = den > 0.f ? (wh * Ou + wb * pb[tid]) / den : 0.f;
  }
}

size_t decode_ws_bytes(const PoolArgs &p, int splits) {
  const int G = p.Hq / p.Hkv;
  return (size_t)p.B * p.Hkv * (splits + 1) * G * PART_STRIDE * sizeof(float);
}

template <int G>
static cudaError_t launch_decode_g(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, int splits,
                                   float *ws, cudaStream_t s) {
  const int pps = (p.max_pages + splits - 1) / splits;
  profile_begin(OSCAR_PROFILE_HISTORY, s);
  hist_partial_kernel<G><<<dim3(splits, p.Hkv, p.B), 128, 0, s>>>(p, q, sm_scale, splits, pps, ws);
  profile_end(OSCAR_PROFILE_HISTORY, s);
  bf16_partial_kernel<G><<<dim3(p.Hkv, p.B), 128, 0, s>>>(p, q, sm_scale, splits, ws);
  const int smem = D * (D + 1) * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(merge_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  merge_kernel<G><<<dim3(p.Hkv, p.B), 128, smem, s>>>(p, splits, ws, out);
  return cudaGetLastError();
}

cudaError_t launch_decode(const PoolArgs &p, const uint16_t *q, float *out, float sm_scale, int splits, float *ws,
                          cudaStream_t s) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_decode_g<1>(p, q, out, sm_scale, splits, ws, s);
    case 2: return launch_decode_g<2>(p, q, out, sm_scale, splits, ws, s);
    case 4: return launch_decode_g<4>(p, q, out, sm_scale, splits, ws, s);
    case 8: return launch_decode_g<8>(p, q, out, sm_scale, splits, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oscar

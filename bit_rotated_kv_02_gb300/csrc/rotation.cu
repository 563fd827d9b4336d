// Rotation construction R = U · H · P and the calibration covariances, in float64 on the GPU.
//
// "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计": the final rotation
// is R = U · Hadamard · bit-reversal; U aligns the directions attention uses (keys: query covariance
// Q^T Q; values: score-weighted value covariance V^T S^T S V), the Hadamard spreads outliers, the
// bit-reversal balances the INT2 groups.  "OSCAR: Offline Spectral Covariance-Aware Rotation for
// 2-bit KV Cache Quantization", Abstract: covariances estimated offline yield fixed rotations.
//
// Conventions (readings): H is the natural-order Sylvester Walsh-Hadamard matrix / sqrt(d); P is the
// bit-reversal permutation, (x · P)[i] = x[bitrev(i)]; Haar U = Q of QR(M) with positive R diagonal;
// covariance U = eigenvectors by descending eigenvalue, each column's largest |entry| positive.
#include "oscar_internal.cuh"
#include "kernels.h"

namespace oscar {

constexpr int RT = 256;  // threads of the one-CTA rotation kernels

__device__ __forceinline__ int bitrev_dev(int i, int bits) { return (int)(__brev((unsigned)i) >> (32 - bits)); }

// Block-wide sum of one double per thread (RT threads).
__device__ double block_sum(double v, double *red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < RT / 32; ++w) t += red[w];
  return t;
}

// ws layout (doubles): [0, d*d) working matrix Q or V; [d*d, d*d + 8) status.
// Haar: Householder QR of M in shared memory (A), Q accumulated in ws, then sign-fixed.
__global__ void __launch_bounds__(RT) haar_kernel(int d, const double *M, double *ws) {
  extern __shared__ double A[];  // [d][d] row-major
  __shared__ double red[RT / 32];
  __shared__ double vk[OSCAR_HEAD_DIM];
  __shared__ double rdiag[OSCAR_HEAD_DIM];
  __shared__ double wcol[OSCAR_HEAD_DIM];
  double *Q = ws;
  const int tid = threadIdx.x;
  for (int i = tid; i < d * d; i += RT) A[i] = M[i];
  __syncthreads();
  // Reflector k: v = x - alpha e1 with alpha = -sign(x0) ||x||, x = A[k:, k]; H_k = I - 2 v v^T / (v^T v).
  // v_k is kept (normalised) in A[k:, k] after R_kk has been recorded in rdiag[k].
  for (int k = 0; k < d; ++k) {
    double part = 0.0;
    for (int i = k + tid; i < d; i += RT) part += A[i * d + k] * A[i * d + k];
    const double nrm2 = block_sum(part, red);
    const double x0 = A[k * d + k];
    const double nrm = sqrt(nrm2);
    const double alpha = (x0 >= 0.0) ? -nrm : nrm;
    const double v0 = x0 - alpha;
    const double vnorm2 = nrm2 - x0 * x0 + v0 * v0;
    __syncthreads();
    if (tid == 0) rdiag[k] = alpha;
    for (int i = k + tid; i < d; i += RT) {
      const double vi = (i == k) ? v0 : A[i * d + k];
      vk[i] = (vnorm2 > 0.0) ? vi / sqrt(vnorm2) : 0.0;
    }
    __syncthreads();
    // A[k:, j] -= 2 v (v^T A[k:, j]) for j > k
    for (int j = k + 1 + tid; j < d; j += RT) {
      double w = 0.0;
      for (int i = k; i < d; ++i) w += vk[i] * A[i * d + j];
      wcol[j] = 2.0 * w;
    }
    __syncthreads();
    for (int idx = tid; idx < (d - k) * (d - k - 1); idx += RT) {
      const int i = k + idx / (d - k - 1), j = k + 1 + idx % (d - k - 1);
      A[i * d + j] -= vk[i] * wcol[j];
    }
    __syncthreads();
    for (int i = k + tid; i < d; i += RT) A[i * d + k] = vk[i];
    __syncthreads();
  }
  // Q = H_0 H_1 ... H_{d-1}: start from I and apply reflectors from the last to the first.
  for (int i = tid; i < d * d; i += RT) Q[i] = (i / d == i % d) ? 1.0 : 0.0;
  __syncthreads();
  for (int k = d - 1; k >= 0; --k) {
    for (int j = tid; j < d; j += RT) {
      double w = 0.0;
      for (int i = k; i < d; ++i) w += A[i * d + k] * Q[i * d + j];
      wcol[j] = 2.0 * w;
    }
    __syncthreads();
    for (int idx = tid; idx < (d - k) * d; idx += RT) {
      const int i = k + idx / d, j = idx % d;
      Q[i * d + j] -= A[i * d + k] * wcol[j];
    }
    __syncthreads();
  }
  // sign fix: column j times sign(R_jj)
  for (int idx = tid; idx < d * d; idx += RT) {
    const int j = idx % d;
    if (rdiag[j] < 0.0) Q[idx] = -Q[idx];
  }
}

// Cyclic Jacobi with the round-robin parallel ordering (d/2 disjoint pairs per round, d-1 rounds
// per sweep).  A in shared memory, eigenvectors accumulated in ws ([d][d], columns), then sorted
// by descending eigenvalue and sign-fixed in place into ws.
__global__ void __launch_bounds__(RT) jacobi_kernel(int d, const double *M, double *ws, int max_sweeps) {
  extern __shared__ double A[];
  __shared__ double cs[OSCAR_HEAD_DIM / 2], sn[OSCAR_HEAD_DIM / 2];
  __shared__ int pp[OSCAR_HEAD_DIM / 2], qq[OSCAR_HEAD_DIM / 2];
  __shared__ double red[RT / 32];
  __shared__ int order[OSCAR_HEAD_DIM];
  __shared__ double evals[OSCAR_HEAD_DIM];
  double *V = ws;
  double *status = ws + d * d;
  const int tid = threadIdx.x;
  const int half = d / 2;
  for (int i = tid; i < d * d; i += RT) {
    // symmetrise the input so that both triangles agree exactly
    const int r = i / d, c = i % d;
    A[i] = 0.5 * (M[r * d + c] + M[c * d + r]);
    V[i] = (r == c) ? 1.0 : 0.0;
  }
  __syncthreads();
  double fro = 0.0;
  {
    double part = 0.0;
    for (int i = tid; i < d * d; i += RT) part += A[i] * A[i];
    fro = sqrt(block_sum(part, red));
  }
  int converged = 0;
  int sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
    double part = 0.0;
    for (int i = tid; i < d * d; i += RT)
      if (i / d != i % d) part += A[i] * A[i];
    const double off = sqrt(block_sum(part, red));
    if (off <= 1e-15 * fro || fro == 0.0) { converged = 1; break; }
    for (int round = 0; round < d - 1; ++round) {
      if (tid < half) {
        // circle method: index d-1 is fixed; pair k joins (round+k, round-k) mod (d-1)
        const int m = d - 1;
        const int a = (round + tid) % m;
        const int b = (tid == 0) ? m : (round - tid + m) % m;
        const int p = min(a, b), q = max(a, b);
        pp[tid] = p; qq[tid] = q;
        const double apq = A[p * d + q];
        double c = 1.0, s = 0.0;
        if (apq != 0.0 && fabs(apq) > 1e-300) {
          const double tau = (A[q * d + q] - A[p * d + p]) / (2.0 * apq);
          const double t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
          c = 1.0 / sqrt(1.0 + t * t);
          s = t * c;
        }
        cs[tid] = c; sn[tid] = s;
      }
      __syncthreads();
      // A <- A J (columns p, q) and V <- V J
      for (int idx = tid; idx < half * d; idx += RT) {
        const int k = idx / d, r = idx % d;
        const int p = pp[k], q = qq[k];
        const double c = cs[k], s = sn[k];
        const double ap = A[r * d + p], aq = A[r * d + q];
        A[r * d + p] = c * ap - s * aq;
        A[r * d + q] = s * ap + c * aq;
        const double vp = V[r * d + p], vq = V[r * d + q];
        V[r * d + p] = c * vp - s * vq;
        V[r * d + q] = s * vp + c * vq;
      }
      __syncthreads();
      // A <- J^T A (rows p, q)
      for (int idx = tid; idx < half * d; idx += RT) {
        const int k = idx / d, col = idx % d;
        const int p = pp[k], q = qq[k];
        const double c = cs[k], s = sn[k];
        const double ap = A[p * d + col], aq = A[q * d + col];
        A[p * d + col] = c * ap - s * aq;
        A[q * d + col] = s * ap + c * aq;
      }
      __syncthreads();
    }
  }
  // order by descending eigenvalue (stable), then sign rule, in place through shared scratch A
  if (tid == 0) {
    for (int i = 0; i < d; ++i) { evals[i] = A[i * d + i]; order[i] = i; }
    for (int i = 1; i < d; ++i) {  // stable insertion sort, descending
      const int oi = order[i];
      int j = i - 1;
      while (j >= 0 && evals[order[j]] < evals[oi]) { order[j + 1] = order[j]; --j; }
      order[j + 1] = oi;
    }
    status[0] = converged ? 1.0 : 0.0;
    status[1] = (double)sweep;
  }
  __syncthreads();
  for (int i = tid; i < d * d; i += RT) A[i] = V[(i / d) * d + order[i % d]];
  __syncthreads();
  for (int j = tid; j < d; j += RT) {
    int best = 0;
    double bv = -1.0;
    for (int i = 0; i < d; ++i)
      if (fabs(A[i * d + j]) > bv) { bv = fabs(A[i * d + j]); best = i; }
    const double sgn = A[best * d + j] < 0.0 ? -1.0 : 1.0;
    for (int i = 0; i < d; ++i) V[i * d + j] = sgn * A[i * d + j];
  }
}

// R = U · H · P: row i of U·H is the natural-order fast Walsh-Hadamard transform of row i of U,
// scaled by 1/sqrt(d); column j of R takes column bitrev(j) of U·H.
__global__ void __launch_bounds__(RT) compose_kernel(int d, const double *U, double *R64, float *R32) {
  extern __shared__ double W[];  // [d][d]
  const int tid = threadIdx.x;
  for (int i = tid; i < d * d; i += RT) W[i] = U[i];
  __syncthreads();
  for (int h = 1; h < d; h <<= 1) {
    for (int idx = tid; idx < d * d / 2; idx += RT) {
      const int row = idx / (d / 2), k = idx % (d / 2);
      const int lo = (k / h) * 2 * h + (k % h), hi = lo + h;
      const double a = W[row * d + lo], b = W[row * d + hi];
      W[row * d + lo] = a + b;
      W[row * d + hi] = a - b;
    }
    __syncthreads();
  }
  const int bits = 31 - __clz(d);
  const double inv = 1.0 / sqrt((double)d);
  for (int idx = tid; idx < d * d; idx += RT) {
    const int i = idx / d, j = idx % d;
    const double r = W[i * d + bitrev_dev(j, bits)] * inv;
    if (R64) R64[idx] = r;
    if (R32) R32[idx] = __double2float_rn(r);
  }
}

size_t rotation_ws_bytes(int d) { return ((size_t)d * d + 8) * sizeof(double); }

cudaError_t launch_make_rotation(int d, int mode, const double *M, double *R64, float *R32, void *ws, cudaStream_t s) {
  double *w = static_cast<double *>(ws);
  const int smem = d * d * (int)sizeof(double);
  cudaError_t e;
  if (mode == OSCAR_ROT_HAAR) {
    if ((e = cudaFuncSetAttribute(haar_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    haar_kernel<<<1, RT, smem, s>>>(d, M, w);
  } else {
    if ((e = cudaFuncSetAttribute(jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    jacobi_kernel<<<1, RT, smem, s>>>(d, M, w, 40);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  compose_kernel<<<1, RT, smem, s>>>(d, w, R64, R32);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// Calibration covariances (float64).
// Generic tiled float64 GEMM: C[M][N] = beta*C + sum_k A(m,k) B(k,n) with element accessors by
// strides (so transposes are free).  16x16 tiles, one output per thread.
__global__ void dgemm_kernel(int Mr, int Nc, int K, const double *A, long sam, long sak, const double *B, long sbk,
                             long sbn, double *C, long scm, double beta) {
  __shared__ double As[16][17], Bs[16][17];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int m = blockIdx.y * 16 + ty, n = blockIdx.x * 16 + tx;
  double acc = 0.0;
  for (int k0 = 0; k0 < K; k0 += 16) {
    As[ty][tx] = (m < Mr && k0 + tx < K) ? A[m * sam + (long)(k0 + tx) * sak] : 0.0;
    Bs[ty][tx] = (n < Nc && k0 + ty < K) ? B[(long)(k0 + ty) * sbk + n * sbn] : 0.0;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) acc += As[ty][k] * Bs[k][tx];
    __syncthreads();
  }
  if (m < Mr && n < Nc) C[m * scm + n] = (beta == 0.0 ? 0.0 : beta * C[m * scm + n]) + acc;
}

static void dgemm(int Mr, int Nc, int K, const double *A, long sam, long sak, const double *B, long sbk, long sbn,
                  double *C, long scm, double beta, cudaStream_t s) {
  dgemm_kernel<<<dim3((Nc + 15) / 16, (Mr + 15) / 16), dim3(16, 16), 0, s>>>(Mr, Nc, K, A, sam, sak, B, sbk, sbn, C,
                                                                           scm, beta);
}

// bf16 [T][heads][d] head h (or [T][d] when heads == 1) -> float64 [T][d]
__global__ void widen_kernel(int64_t T, int heads, int h, int d, const uint16_t *x, double *y) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < T * d; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / d;
    const int c = (int)(i % d);
    y[i] = (double)bf16_to_f32(x[(t * heads + h) * d + c]);
  }
}

// Causal row softmax of S [T][T] in place (one warp per row); entries above the diagonal -> 0.
__global__ void causal_softmax_kernel(int64_t T, double scale, double *S) {
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  double *row = S + t * T;
  double mx = -INFINITY;
  for (int64_t u = lane; u <= t; u += 32) mx = fmax(mx, row[u] * scale);
  for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(FULL, mx, o));
  double sum = 0.0;
  for (int64_t u = lane; u <= t; u += 32) sum += exp(row[u] * scale - mx);
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
  for (int64_t u = lane; u < T; u += 32) row[u] = (u <= t) ? exp(row[u] * scale - mx) / sum : 0.0;
}

// C = sum over (t, h) of Q[t][h]^T Q[t][h]: the [T*heads][d] rows form one tall matrix.
__global__ void cov_k_kernel(int64_t T, int heads, int d, const uint16_t *Q, double *C) {
  __shared__ double Ai[16][17], Aj[16][17];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int i = blockIdx.y * 16 + ty, j = blockIdx.x * 16 + tx;
  const int64_t rows = T * heads;
  double acc = 0.0;
  for (int64_t r0 = 0; r0 < rows; r0 += 16) {
    // Ai[rr][c] = Q[r0+rr][blockIdx.y*16 + c], Aj[rr][c] = Q[r0+rr][blockIdx.x*16 + c]
    const int64_t r = r0 + ty;
    const int ci = blockIdx.y * 16 + tx, cj = blockIdx.x * 16 + tx;
    Ai[ty][tx] = (r < rows && ci < d) ? (double)bf16_to_f32(Q[r * d + ci]) : 0.0;
    Aj[ty][tx] = (r < rows && cj < d) ? (double)bf16_to_f32(Q[r * d + cj]) : 0.0;
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) acc += Ai[rr][ty] * Aj[rr][tx];
    __syncthreads();
  }
  if (i < d && j < d) C[i * d + j] = acc;
}

cudaError_t launch_cov_k(int64_t T, int heads, int d, const uint16_t *Q, double *C, cudaStream_t s) {
  cov_k_kernel<<<dim3((d + 15) / 16, (d + 15) / 16), dim3(16, 16), 0, s>>>(T, heads, d, Q, C);
  return cudaGetLastError();
}

size_t cov_v_ws_bytes(int64_t T, int d) { return ((size_t)T * T + 4 * (size_t)T * d) * sizeof(double); }

cudaError_t launch_cov_v(int64_t T, int heads, int d, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                         double scale, double *C, void *ws, cudaStream_t s) {
  double *S = static_cast<double *>(ws);
  double *Qh = S + T * T, *Kd = Qh + T * d, *Vd = Kd + T * d, *O = Vd + T * d;
  const int wb = 1024;
  widen_kernel<<<wb, 256, 0, s>>>(T, 1, 0, d, K, Kd);
  widen_kernel<<<wb, 256, 0, s>>>(T, 1, 0, d, V, Vd);
  for (int h = 0; h < heads; ++h) {
    widen_kernel<<<wb, 256, 0, s>>>(T, heads, h, d, Q, Qh);
    dgemm((int)T, (int)T, d, Qh, d, 1, Kd, 1, d, S, T, 0.0, s);            // S = Qh K^T
    causal_softmax_kernel<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(T, scale, S);
    dgemm((int)T, d, (int)T, S, T, 1, Vd, d, 1, O, d, 0.0, s);             // O = S V
    dgemm(d, d, (int)T, O, 1, d, O, d, 1, C, d, h == 0 ? 0.0 : 1.0, s);    // C (+)= O^T O
  }
  return cudaGetLastError();
}

}  // namespace oscar

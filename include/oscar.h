/*
 * oscar.h — C ABI of the GB300 (sm_103a) OSCAR INT2 KV-cache library (liboscar.so).
 *
 * OSCAR keeps a three-segment KV pool per sequence and layer:
 *     BF16 sink (64 tokens) | rotated INT2 history (paged) | BF16 recent (256 tokens)
 * ("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计";
 *  "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract).
 * History vectors are rotated by a fixed orthogonal R = U · H · P, clipped, quantized per group
 * to 2-bit codes with a bf16 scale and zero point, and packed 4 codes per byte.
 *
 * Conventions shared by every call
 *   - Every tensor argument is a DEVICE pointer owned by the caller (unless stated otherwise).
 *     The library never allocates or frees memory; scratch space comes from a caller-provided
 *     workspace whose size a *_workspace_size() query returns.
 *   - bf16 values are passed as raw 16-bit patterns (oscar_bf16).
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL = legacy default stream)
 *     unless stated otherwise.  Arguments are validated on the host before any launch; an invalid
 *     call launches nothing and returns an error status.
 *   - Errors that can only be seen on the device (a page-table entry outside the page pool, a
 *     history that would overflow its page-table row, bookkeeping counters out of range) never
 *     fault: the kernel skips the affected access and ORs an OSCAR_DEVERR_* bit into pool->err.
 *   - oscar_last_error_string() describes the last failure of the calling thread.
 *   - Vectors are rows: a head vector x (1 x d) is rotated as x_rot = x · R; R arrays are
 *     row-major [d][d] float32.
 *   - Only head_dim 128, group sizes 32/64/128 and Hq/Hkv in {1, 2, 4, 8} are supported.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum oscar_status {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1,  /* null pointer, inconsistent sizes, bad mode                 */
  OSCAR_ERR_UNSUPPORTED = 2,  /* head_dim != 128, group size not 32/64/128, GQA ratio > 8   */
  OSCAR_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the size query returned  */
  OSCAR_ERR_CUDA = 4,         /* a CUDA runtime error (see oscar_last_error_string)         */
  OSCAR_ERR_NUMERIC = 5       /* the eigensolver did not converge                           */
} oscar_status_t;

typedef uint16_t oscar_bf16;   /* raw bf16 bit pattern */
typedef void *oscar_stream_t;  /* cudaStream_t */

#define OSCAR_HEAD_DIM 128
#define OSCAR_PAGE_TOKENS 64
#define OSCAR_SINK_TOKENS 64
#define OSCAR_RECENT_TOKENS 256

/* Device-side error bits (OR-ed into pool->err; the affected access is skipped). */
#define OSCAR_DEVERR_PAGE_INDEX 1u   /* page-table entry outside [0, num_pages)          */
#define OSCAR_DEVERR_HISTORY_FULL 2u /* hist_len would exceed max_pages * 64             */
#define OSCAR_DEVERR_COUNTERS 4u     /* sink_len/recent_start/recent_len/hist_len invalid */
#define OSCAR_DEVERR_TIMEOUT 8u      /* an internal pipeline wait exceeded its time limit   */
#define OSCAR_DEVERR_DEBUG_CHECK 16u /* debug build only (liboscar_debug.so, compiled with OSCAR_DEBUG):
                                        a device-side bounds check of a workspace, partial-slot or pool
                                        index failed; the access was skipped                 */

/* Rotation construction modes for oscar_make_rotation. */
#define OSCAR_ROT_HAAR 0        /* M = d x d standard-normal draws; U = Q of QR(M), sign-fixed */
#define OSCAR_ROT_COVARIANCE 1  /* M = d x d symmetric covariance; U = eigenvectors            */

/*
 * The three-segment pool of one layer (a plain struct of device pointers and sizes).
 * Layouts (row-major, innermost last):
 *   sink_k, sink_v          bf16  [batch][Hkv][64][d]
 *   recent_k, recent_v      bf16  [batch][Hkv][256][d]   ring buffer
 *   codes_k, codes_v        u8    [num_pages][Hkv][64][d/4]   channel 4b+i -> byte b, bits 2i..2i+1
 *   scale_k/zero_k/scale_v/zero_v
 *                           bf16  [num_pages][Hkv][64][d/group_size]
 *   page_table              int32 [batch][max_pages]   physical page of history page i of sequence b
 *   sink_len, hist_len, recent_start, recent_len   int32 [batch]
 *   R_k, R_v                fp32  [Hkv][d][d]   rotation of keys / values (x_rot = x · R)
 *   clip_k, clip_v          fp32  [Hkv]         clip ratios in (0, 1]
 *   codebook_k, codebook_v  fp32  [Hkv][4]      optional (NULL = uniform INT2): the four dequantization
 *                                               levels l0 < l1 < l2 < l3 of a Lloyd-Max codebook in the
 *                                               group's coordinate t = (x_rot - zero) / scale; a code is the
 *                                               nearest level (ties to the even code) and dequantizes to
 *                                               zero + scale * l[code]; 16-byte aligned.  With group
 *                                               size 128 the tensor-core attention takes the codes'
 *                                               indicator planes [c >= i] (three MMAs where the uniform
 *                                               levels need one); other group sizes decode on the
 *                                               CUDA-core path with a 4-entry table.
 *   err                     uint32 [1]          device error word (OSCAR_DEVERR_* bits)
 *   sync                    int32 [batch]       arrival counters; zero them once before the first
 *                                               call, every call leaves them zero again
 * Every array of the pool is 16-byte aligned (the decode kernels move pages with bulk asynchronous copies).
 * Token placement: positions 0..63 -> sink; later tokens -> recent slot
 * (recent_start + recent_len) % 256; the oldest recent token (slot recent_start) is demoted to
 * history position hist_len: page page_table[b][hist_len / 64], row hist_len % 64.
 */
typedef struct oscar_pool {
  int32_t batch, num_q_heads, num_kv_heads, head_dim, group_size;
  int32_t num_pages, max_pages;
  oscar_bf16 *sink_k, *sink_v;
  oscar_bf16 *recent_k, *recent_v;
  uint8_t *codes_k, *codes_v;
  oscar_bf16 *scale_k, *zero_k, *scale_v, *zero_v;
  int32_t *page_table;
  int32_t *sink_len, *hist_len, *recent_start, *recent_len;
  const float *R_k, *R_v;
  const float *clip_k, *clip_v;
  uint32_t *err;
  int32_t *sync;
  const float *codebook_k, *codebook_v;
} oscar_pool;

/* Description of the calling thread's last error ("" if none). Never NULL. */
const char *oscar_last_error_string(void);

/* Library version string. */
const char *oscar_version(void);

/*
 * Rotation construction R = U · H · P ("OSCAR 的设计": R = U · Hadamard · bit-reversal; U from the
 * query covariance Q^T Q for keys and the score-weighted value covariance V^T S^T S V for values;
 * Abstract: fixed rotations derived offline from attention-aware covariances).
 *   d        head dimension (128; any power of two 2..128 is accepted for testing)
 *   mode     OSCAR_ROT_HAAR: M holds d x d standard-normal draws, U = Q of the QR decomposition
 *            of M with columns multiplied by sign(diag(R_qr));
 *            OSCAR_ROT_COVARIANCE: M is a symmetric covariance, U = its eigenvectors ordered by
 *            descending eigenvalue, each column signed so its largest-magnitude entry is positive.
 *   M        device fp64 [d][d] (row-major), read only
 *   R64      device fp64 [d][d] output (may be NULL)
 *   R32      device fp32 [d][d] output, each entry the nearest float32 to R64 (may be NULL)
 *   ws       device workspace of at least oscar_make_rotation_workspace_size(d) bytes
 * H is the natural-order Walsh-Hadamard matrix / sqrt(d); P the bit-reversal permutation,
 * (x · P)[i] = x[bitrev(i)].  Runs in float64 on one CTA.  SYNCHRONOUS: waits for the stream and
 * returns OSCAR_ERR_NUMERIC if the Jacobi eigensolver did not converge.
 */
size_t oscar_make_rotation_workspace_size(int32_t d);
oscar_status_t oscar_make_rotation(int32_t d, int32_t mode, const double *M, double *R64, float *R32,
                                   void *ws, size_t ws_bytes, oscar_stream_t stream);

/*
 * Calibration covariances (offline; "OSCAR 的设计": keys use Q^T Q, values V^T S^T S V).
 *   oscar_calib_covariance_k: C = sum over heads h of Q_h^T Q_h, Q bf16 [T][heads][d].
 *   oscar_calib_covariance_v: C = sum over heads h of (S_h V)^T (S_h V), S_h the causal row
 *       softmax of Q_h K^T * softmax_scale; Q bf16 [T][heads][d], K and V bf16 [T][d].
 *   C: device fp64 [d][d] output.  float64 arithmetic.  Asynchronous.
 */
oscar_status_t oscar_calib_covariance_k(int64_t T, int32_t heads, int32_t d, const oscar_bf16 *Q, double *C,
                                        oscar_stream_t stream);
size_t oscar_calib_covariance_v_workspace_size(int64_t T, int32_t heads, int32_t d);
oscar_status_t oscar_calib_covariance_v(int64_t T, int32_t heads, int32_t d, const oscar_bf16 *Q,
                                        const oscar_bf16 *K, const oscar_bf16 *V, double softmax_scale,
                                        double *C, void *ws, size_t ws_bytes, oscar_stream_t stream);

/*
 * Bulk rotate / clip / quantize / pack of many head vectors ("OSCAR 的设计": rotate, clip,
 * quantize and pack, 4 two-bit values per byte; the long middle of a prompt becomes INT2 history).
 *   x       bf16 [n_tokens][Hkv][d]          input rows
 *   R32     fp32 [Hkv][d][d]                 per-head rotation
 *   clip    fp32 [Hkv]                       per-head clip ratio c in (0, 1]
 *   codes   u8   [n_tokens][Hkv][d/4]        output
 *   scale, zero  bf16 [n_tokens][Hkv][d/group_size]  output
 *   stats   uint32 [4] or NULL: [0] += elements re-evaluated exactly, [1] += groups whose scale/zero
 *           needed the exact path, [2] += results not proven correctly rounded (expected 0),
 *           [3] |= OSCAR_DEVERR_* bits of device-side failures (a pipeline wait that timed out)
 *   Alignment: x, R32 and codes 16 bytes; scale and zero 8 bytes.
 * Arithmetic per group (IEEE float32, nearest-even): x_hat = nearest float32 to the exact x · R;
 * lo = c*min, hi = c*max, s = (hi-lo)/3, scale = bf16(s), zero = bf16(lo),
 * code = clamp(rint((x_hat - zero)/scale), 0, 3) with the stored bf16 scale/zero; scale 0 -> codes 0.
 * The rotation runs on the tensor cores; elements whose rounding the fast result cannot decide are
 * re-evaluated exactly.
 */
oscar_status_t oscar_quantize_kv(int64_t n_tokens, int32_t num_kv_heads, int32_t head_dim, int32_t group_size,
                                 const oscar_bf16 *x, const float *R32, const float *clip, uint8_t *codes,
                                 oscar_bf16 *scale, oscar_bf16 *zero, uint32_t *stats, oscar_stream_t stream);

/*
 * oscar_quantize_kv with a codebook: the same rotation, scale and zero, and for each element the
 * nearest of the four levels codebook[h][0..3] (float32, strictly increasing) to t = (x_hat - zero) / scale
 * in float32, ties to the even code (midpoints m_i = (l_i + l_{i+1}) * 0.5 in float32;
 * code = #{i : t > m_i} + (t == m_1)).  The levels (0, 1, 2, 3) give oscar_quantize_kv's codes.
 *   codebook fp32 [Hkv][4], 16-byte aligned.  The rotation runs on the CUDA cores.
 */
oscar_status_t oscar_quantize_kv_codebook(int64_t n_tokens, int32_t num_kv_heads, int32_t head_dim,
                                          int32_t group_size, const oscar_bf16 *x, const float *R32,
                                          const float *clip, const float *codebook, uint8_t *codes,
                                          oscar_bf16 *scale, oscar_bf16 *zero, uint32_t *stats,
                                          oscar_stream_t stream);

/*
 * Lloyd-Max calibration of a 4-level codebook per KV head ("超越TurboQuant！OSCAR：面向真实服务的2-bit
 * KV Cache量化", closing comparison with TurboQuant: a Lloyd-Max codebook on top of the rotation).
 * For the calibration rows x bf16 [n][Hkv][d] (keys or values), R32 fp32 [Hkv][d][d], clip fp32 [Hkv]:
 * every element's t = (x_rot - zero) / scale with the uniform quantizer's bf16 scale and zero (x_rot by
 * float32 FMA dots; groups with a zero or non-finite scale are left out), then Lloyd's method per head
 * from the levels (0, 1, 2, 3): cells by the nearest level (ties to the even code, float64 midpoints),
 * each level moved to its cell's mean (an empty cell keeps its level), until no level moves or
 * max_iters iterations.  codebook: fp32 [Hkv][4] output.  ws: device scratch of at least
 * oscar_lloyd_max_workspace_size bytes, 16-byte aligned.  x and R32 16-byte aligned.
 */
oscar_status_t oscar_lloyd_max_workspace_size(int64_t n, int32_t num_kv_heads, size_t *bytes);
oscar_status_t oscar_lloyd_max_codebook(int64_t n, int32_t num_kv_heads, int32_t head_dim, int32_t group_size,
                                        const oscar_bf16 *x, const float *R32, const float *clip,
                                        int32_t max_iters, float *codebook, void *ws, size_t ws_bytes,
                                        oscar_stream_t stream);

/*
 * Bulk prefill of one sequence into the pool: tokens [0, 64) -> sink, [64, len-256) -> history
 * (quantized as in oscar_quantize_kv, written through page_table[seq]), [len-256, len) -> recent
 * (recent_start = 0).  k, v: bf16 [len][Hkv][d].  Sets sink_len/hist_len/recent_start/recent_len
 * of `seq`.  page_table[seq] must hold ceil((len-320)/64) valid pages.
 */
oscar_status_t oscar_prefill_pool(const oscar_pool *pool, int32_t seq, int64_t len, const oscar_bf16 *k,
                                  const oscar_bf16 *v, uint32_t *stats, oscar_stream_t stream);

/*
 * Bulk prefill of a sequence whose prompt starts with the same tokens as a sequence already in the
 * pool (a shared prefix: the paged, prefix-cache-compatible history of the Abstract and of "OSCAR 的
 * 设计"; "评估结果" Fig. 6 measures the prefix-cache hit ratio).  As oscar_prefill_pool, except that
 * the first `shared_pages` history pages are taken as already in place: page_table[seq][0 ..
 * shared_pages) points at pages written for the other sequence (the same physical pages), and those
 * pages are neither quantized nor written.  Only whole pages can be shared (shared_pages * 64 <=
 * history length); demotions write only at and after the history length, so shared pages are never
 * written again.  k and v still hold all `len` tokens (the sink and recent window are per sequence).
 */
oscar_status_t oscar_prefill_pool_shared(const oscar_pool *pool, int32_t seq, int64_t len, const oscar_bf16 *k,
                                         const oscar_bf16 *v, int32_t shared_pages, uint32_t *stats,
                                         oscar_stream_t stream);

/*
 * Demotion ("OSCAR 的设计": the oldest recent token is rotated, clipped, quantized and packed by a
 * fused kernel and demoted into the INT2 history).
 * For every sequence whose recent window is full (recent_len == 256) — or, if mask (device int32
 * [batch]) is not NULL, every sequence with mask[b] != 0 and recent_len > 0 — the K and V vectors
 * in recent slot recent_start are quantized into history position hist_len of every KV head;
 * then hist_len += 1, recent_start = (recent_start + 1) % 256, recent_len -= 1.
 * The page for the new position must already be in page_table (else OSCAR_DEVERR_* and the
 * sequence is left unchanged).
 */
oscar_status_t oscar_demote(const oscar_pool *pool, const int32_t *mask, oscar_stream_t stream);

/*
 * Append one new token per sequence ("OSCAR 的设计": a new token is first written into the recent
 * window).  Demotes first where the recent window is full (as oscar_demote with mask NULL), then
 * writes k_new/v_new (bf16 [batch][Hkv][d]) to the sink while it holds fewer than 64 tokens and the
 * rest of the pool is empty, else to recent slot (recent_start + recent_len) % 256.  One launch.
 */
oscar_status_t oscar_append_kv(const oscar_pool *pool, const oscar_bf16 *k_new, const oscar_bf16 *v_new,
                               oscar_stream_t stream);

/*
 * Decode attention over the pool ("OSCAR 的设计": the INT2 kernel unpacks, dequantizes with
 * scale/zero point and accumulates in floating point; a BF16 kernel handles sink/recent; an online
 * softmax merge combines the two.  Abstract: a custom INT2 attention kernel compatible with paged
 * KV-cache serving).
 *   q       bf16 [batch][Hq][d]; query head h reads KV head h / (Hq/Hkv)
 *   out     fp32 [batch][Hq][d]
 *           q and out (and k_new, v_new of the calls that take them) are read and written by the kernels
 *           themselves: device (or managed) memory, or page-locked host memory mapped into the device's
 *           address space at the same address (cudaHostAlloc under unified addressing), which the kernels
 *           then access over the host link with no separate copy.  Other pointers (pageable host memory)
 *           are refused with OSCAR_ERR_INVALID_ARG before any launch.
 *   softmax_scale   > 0 (usually 1/sqrt(d))
 *   num_splits      history split factor per (sequence, KV head) for pools with a codebook and group
 *                   size 32/64; 0 = choose to fill the GPU.  Every other pool balances the history
 *                   pages of all (sequence, KV head) pairs over a GPU-filling grid itself and ignores it.
 *   ws, ws_bytes    workspace, 16-byte aligned: oscar_decode_workspace_size() bytes (same pool shape and
 *                   num_splits) enable every part of the decode; a smaller one down to the pool's minimum
 *                   is accepted (group size 128 then splits the history statically, without the dynamic
 *                   tail in which CTAs that finish early take the remaining pages), less is refused with
 *                   OSCAR_ERR_WORKSPACE
 * out[b][h] = sum over all pool tokens of softmax(score) * value, with score = q·k*scale for sink
 * and recent tokens and (q·R_k)·k_rot*scale for history tokens, whose values enter as v_rot·R_v^T.
 * Kernels: uniform pools of group size 128 run the warp-MMA history kernel, uniform pools of group
 * size 32/64 the tensor-memory (tcgen05) history kernel, codebook pools of group size 32/64 the CUDA-core
 * kernels.  The environment variable OSCAR_DECODE_TC=1 (read once per process) routes uniform pools of
 * group size 128 to the tensor-memory kernel too (for comparison and tests; same results up to float32
 * rounding).
 */
oscar_status_t oscar_decode_workspace_size(const oscar_pool *pool, int32_t num_splits, size_t *bytes);
oscar_status_t oscar_decode_attention(const oscar_pool *pool, const oscar_bf16 *q, float *out, float softmax_scale,
                                      int32_t num_splits, void *ws, size_t ws_bytes, oscar_stream_t stream);

/*
 * One decode step: oscar_append_kv(pool, k_new, v_new) followed by oscar_decode_attention(pool, q,
 * out, softmax_scale, 0, ws, ws_bytes): the same pool afterwards, byte for byte, and the same
 * attention output up to float32 rounding ("OSCAR 的设计": the new token enters the recent window,
 * the oldest recent token is demoted into the INT2 history, then attention runs over the three
 * segments).  With group size 128 the attention runs over the history before the step and the BF16
 * window after the append; the attention kernel's sink CTAs perform the demotion
 * and add the demoted token as a partial, the merge kernel stores the new token and advances the
 * counters; uniform pools of group size 32/64 do the same around the tensor-memory history kernel.
 * Codebook pools of group size 32/64 run the two calls in turn.
 *   k_new, v_new   bf16 [batch][Hkv][d] (16-byte aligned); q bf16 [batch][Hq][d] (16-byte aligned)
 *   ws, ws_bytes   at least oscar_decode_workspace_size(pool, 0) bytes
 * Errors as for the two calls; all checks run before any launch.
 */
oscar_status_t oscar_decode_step(const oscar_pool *pool, const oscar_bf16 *k_new, const oscar_bf16 *v_new,
                                 const oscar_bf16 *q, float *out, float softmax_scale, void *ws, size_t ws_bytes,
                                 oscar_stream_t stream);

/*
 * Kernel timing hook (measurement support; no counterpart on the pages).  Arms the calling thread so
 * that its next call that launches the kernel of kind `which` records cudaEvent_t `start` on the call's
 * stream immediately before that kernel and `stop` immediately after it, then disarms.
 *   which = OSCAR_PROFILE_HISTORY: the INT2 history kernel of oscar_decode_attention;
 *   which = OSCAR_PROFILE_DEMOTE:  the demote/append kernel of oscar_demote / oscar_append_kv.
 * Passing NULL events disarms.  The events are owned by the caller.
 */
#define OSCAR_PROFILE_HISTORY 0
#define OSCAR_PROFILE_DEMOTE 1
oscar_status_t oscar_profile_events(int32_t which, void *start, void *stop);

/*
 * Allocation-free decode attention (no counterpart on the pages: an interface convenience).
 * Some callers cannot call cudaMalloc: a serving engine that has already handed all device memory to
 * its KV pool and activation arenas, or a latency-critical decode loop that must not block on the
 * device allocator (cudaMalloc may synchronize the device).  This entry point computes exactly what
 * oscar_decode_attention(pool, q, out, softmax_scale, 0, ws, ...) computes, but its scratch space is a
 * fixed device array of OSCAR_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU that loads
 * the library holds that array until the process exits.  It calls no allocator.
 *   - Pools whose decode workspace (oscar_decode_workspace_size with num_splits 0) exceeds
 *     OSCAR_NOALLOC_SCRATCH_BYTES are rejected with OSCAR_ERR_WORKSPACE before any launch.
 *   - The first call on each device looks the array's device address up (cudaGetSymbolAddress) with
 *     that device current; make that first call before starting any stream capture.  A device reset
 *     (cudaDeviceReset) ends the context the address belongs to: the first call in the new context looks
 *     it up again (the calls key the address by the current context's identifier).
 *   - All calls share the one array, and each call writes every scratch word it later reads, so
 *     nothing needs clearing; but two calls whose kernels overlap on the GPU (different streams, or
 *     different host threads) race on it.  Order such calls on one stream.
 */
#define OSCAR_NOALLOC_SCRATCH_BYTES (8u << 20)
oscar_status_t oscar_decode_attention_noalloc(const oscar_pool *pool, const oscar_bf16 *q, float *out,
                                              float softmax_scale, oscar_stream_t stream);

/*
 * BF16 paged KV cache: the comparison baseline ("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化",
 * section "评估结果", Fig. 5, and the arXiv listing's Abstract: batch-1 decoding at 100k context is up
 * to about 3x faster with the INT2 history than with the history kept in BF16, because fewer KV bytes
 * are read).  Every token of a sequence is kept in BF16, in 64-token pages, as a paged serving engine
 * keeps it; these calls let both sides of that comparison run on the same GPU.
 * Layouts (row-major, innermost last):
 *   k_pages, v_pages   bf16  [num_pages][Hkv][64][d]   16-byte aligned; token t of sequence b sits at
 *                            page page_table[b][t / 64], row t % 64
 *   page_table         int32 [batch][max_pages]
 *   seq_len            int32 [batch]   tokens held, 0 <= seq_len <= max_pages * 64
 *   err                uint32 [1]      device error word (OSCAR_DEVERR_* bits)
 * Limits: head_dim 128, Hq/Hkv in {1, 2, 4, 8}, num_pages * Hkv * 64 < 2^31.
 */
typedef struct oscar_bf16_cache {
  int32_t batch, num_q_heads, num_kv_heads, head_dim;
  int32_t num_pages, max_pages;
  oscar_bf16 *k_pages, *v_pages;
  int32_t *page_table;
  int32_t *seq_len;
  uint32_t *err;
} oscar_bf16_cache;

/*
 * Bulk prefill of one sequence: k, v bf16 [len][Hkv][d] (16-byte aligned) -> tokens [0, len) of
 * sequence `seq` through page_table[seq]; sets seq_len[seq] = len.  page_table[seq] must hold
 * ceil(len / 64) valid pages (an entry outside [0, num_pages) skips that page and sets
 * OSCAR_DEVERR_PAGE_INDEX).
 */
oscar_status_t oscar_bf16_prefill(const oscar_bf16_cache *cache, int32_t seq, int64_t len, const oscar_bf16 *k,
                                  const oscar_bf16 *v, oscar_stream_t stream);

/*
 * Append one token per sequence: k_new, v_new bf16 [batch][Hkv][d] (16-byte aligned) are written at
 * position seq_len[b] (page page_table[b][seq_len / 64], row seq_len % 64); then seq_len[b] += 1.
 * A full sequence (seq_len == max_pages * 64) sets OSCAR_DEVERR_HISTORY_FULL, a page-table entry
 * outside the pool OSCAR_DEVERR_PAGE_INDEX; that sequence is left unchanged.
 */
oscar_status_t oscar_bf16_append_kv(const oscar_bf16_cache *cache, const oscar_bf16 *k_new, const oscar_bf16 *v_new,
                                    oscar_stream_t stream);

/*
 * Decode attention over the BF16 cache: out[b][h] = sum over the seq_len[b] tokens of
 * softmax(q·k * softmax_scale) * v, query head h reading KV head h / (Hq/Hkv); an empty sequence
 * gives zeros.
 *   q     bf16 [batch][Hq][d] (4-byte aligned);  out  fp32 [batch][Hq][d]
 *   ws    workspace of at least oscar_bf16_decode_workspace_size() bytes (split partials)
 */
oscar_status_t oscar_bf16_decode_workspace_size(const oscar_bf16_cache *cache, size_t *bytes);
oscar_status_t oscar_bf16_decode_attention(const oscar_bf16_cache *cache, const oscar_bf16 *q, float *out,
                                           float softmax_scale, void *ws, size_t ws_bytes, oscar_stream_t stream);

/*
 * One decode step over the BF16 cache: oscar_bf16_append_kv then oscar_bf16_decode_attention, with
 * the same results, launched as one chain.
 */
oscar_status_t oscar_bf16_decode_step(const oscar_bf16_cache *cache, const oscar_bf16 *k_new,
                                      const oscar_bf16 *v_new, const oscar_bf16 *q, float *out,
                                      float softmax_scale, void *ws, size_t ws_bytes, oscar_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */

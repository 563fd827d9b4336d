// Split of the history over the history CTAs of a decode launch: the flattened (sequence, KV head, page)
// space is cut into equal contiguous ranges, chunk = ceil(total / n_hist), CTA i taking [i chunk, (i+1) chunk)
// (with a dynamic tail, below, the ranges cover the static part only).  The merge kernel locates a segment's
// partial slots with the same arithmetic.
#pragma once

#include "oscar_internal.cuh"
#include "ptx.cuh"

namespace oscar {
namespace split {

// hist_len[b], kept in L2 between steps (evict last)
__device__ __forceinline__ int hist_len_of(const PoolArgs &p, int b) { return ld_hint(p.hist_len + b, l2_evict_last()); }

__device__ __forceinline__ int npages_of(const PoolArgs &p, int b) {
  int hl = hist_len_of(p, b);
  hl = max(0, min(hl, p.max_pages * PAGE));
  return (hl + PAGE - 1) / PAGE;
}

// Dynamic tail of the split (group-128 decode, when the caller's workspace holds its partial slots): once
// the history holds at least 64 pages per history CTA, its last tenth is cut into at most 4 n_hist chunks
// of at least 16 pages,
// which the CTAs claim one at a time (an atomic counter) once their own range is done, so that the CTAs an
// SM's other work slowed down hand pages to the faster ones.  The static ranges split the first
// static_pages pages as before; chunk k covers pages [static_pages + k dyn_pages, ... + dyn_pages) (the last
// one may be shorter).  Partial slots: static range of CTA i, segment s: i + s; chunk k, segment s:
// dyn_slot0 + k + s with dyn_slot0 = n_hist + 7 B Hkv (after the BF16 and demoted-token slots).
struct Plan {
  long long total;         // history pages of all (sequence, KV head) segments
  long long static_pages;  // pages of the static ranges
  long long chunk;         // static range length
  long long n_dyn;         // chunks
  long long dyn_pages;     // pages per chunk
};
__host__ __device__ __forceinline__ long long max_dyn_chunks(int n_hist) { return 4LL * n_hist; }
__host__ __device__ __forceinline__ Plan plan_of(long long total, int n_hist, bool dyn) {
  Plan pl;
  pl.total = total;
  const long long td = (dyn && total >= 64LL * n_hist) ? total / 10 : 0;
  pl.static_pages = total - td;
  pl.chunk = (pl.static_pages + n_hist - 1) / n_hist;
  // at least 16 pages a chunk: a claim costs a round of loads (the counter, the position, the page table)
  pl.dyn_pages = td > 0 ? max(16LL, (td + max_dyn_chunks(n_hist) - 1) / max_dyn_chunks(n_hist)) : 1;
  pl.n_dyn = td > 0 ? (td + pl.dyn_pages - 1) / pl.dyn_pages : 0;
  return pl;
}

// Position of flattened page `start` (which must exist): sequence b, KV head kvh, page local of that
// sequence's history, its page count np and history length hl.  Run by one full warp; results in every lane.
static __device__ void locate_at(const PoolArgs &p, long long start, int &b, int &kvh, int &local, int &np, int &hl) {
  const int lane = threadIdx.x & 31;
  const int K = (p.B + 31) / 32, first = min(p.B, lane * K), last = min(p.B, first + K);
  long long bsum = 0;
#pragma unroll 8
  for (int x = first; x < last; ++x) bsum += (long long)npages_of(p, x) * p.Hkv;
  long long inc = bsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(FULL, inc, o);
    if (lane >= o) inc += t;
  }
  const long long excl = inc - bsum;
  const unsigned hit = __ballot_sync(FULL, bsum > 0 && start >= excl && start < excl + bsum);
  int bb = 0, kk = 0, ll = 0, npx0 = 0, hl0 = 0;
  const int src = hit ? __ffs(hit) - 1 : 0;
  if (hit && lane == src) {
    long long run = excl;
    for (int x = first; x < last; ++x) {
      const int hx = max(0, min(hist_len_of(p, x), p.max_pages * PAGE));
      const int npx = (hx + PAGE - 1) / PAGE;
      const long long v = (long long)npx * p.Hkv;
      if (v > 0 && start < run + v) {
        bb = x; kk = (int)((start - run) / npx); ll = (int)((start - run) % npx); npx0 = npx; hl0 = hx;
        break;
      }
      run += v;
    }
  }
  b = __shfl_sync(FULL, bb, src);
  kvh = __shfl_sync(FULL, kk, src);
  local = __shfl_sync(FULL, ll, src);
  np = __shfl_sync(FULL, npx0, src);
  hl = __shfl_sync(FULL, hl0, src);
}

// This CTA's share of the flattened (sequence, KV head, page) space: pages [lo, lo + n) of the static
// ranges (lo = cta * chunk within the plan's static_pages; plan_of with dyn = false: all pages), and the
// position (b0, kvh0, local0) of page lo plus the page count np0 and history length hl0 of sequence b0.
// Run by one full warp; results valid in every lane.  Up to 32 sequences one load of hist_len per lane
// serves everything.
static __device__ void locate_range(const PoolArgs &p, int n_hist, int cta, bool dyn, long long &lo, long long &n,
                                    int &b0, int &kvh0, int &local0, int &np0, int &hl0, Plan &pl) {
  const int lane = threadIdx.x & 31;
  b0 = 0; kvh0 = 0; local0 = 0; np0 = 0; hl0 = 0;
  if (p.B <= 32) {
    const int hl = lane < p.B ? max(0, min(hist_len_of(p, lane), p.max_pages * PAGE)) : 0;
    const int np = (hl + PAGE - 1) / PAGE;
    const long long v = (long long)np * p.Hkv;
    long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += t;
    }
    const long long total = __shfl_sync(FULL, inc, 31);
    pl = plan_of(total, n_hist, dyn);
    lo = (long long)cta * pl.chunk;
    n = max(0ll, min(pl.static_pages, lo + pl.chunk) - lo);
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
  // more than 32 sequences: lane l takes the block of sequences [l K, l K + K), K = ceil(B / 32); the block
  // sums come from one round of independent loads, a warp scan orders the blocks, and the lane whose block
  // holds page lo walks it
  const int K = (p.B + 31) / 32, first = min(p.B, lane * K), last = min(p.B, first + K);
  long long bsum = 0;
#pragma unroll 8
  for (int x = first; x < last; ++x) bsum += (long long)npages_of(p, x) * p.Hkv;
  long long inc = bsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(FULL, inc, o);
    if (lane >= o) inc += t;
  }
  const long long total = __shfl_sync(FULL, inc, 31);
  pl = plan_of(total, n_hist, dyn);
  lo = (long long)cta * pl.chunk;
  n = max(0ll, min(pl.static_pages, lo + pl.chunk) - lo);
  const long long excl = inc - bsum;
  const unsigned hit = __ballot_sync(FULL, bsum > 0 && lo >= excl && lo < excl + bsum);
  if (n > 0 && hit) {
    const int src = __ffs(hit) - 1;
    int bb = 0, kk = 0, ll = 0, np = 0, hl = 0;
    if (lane == src) {
      long long run = excl;
      for (int x = first; x < last; ++x) {
        const int hx = max(0, min(hist_len_of(p, x), p.max_pages * PAGE));
        const int npx = (hx + PAGE - 1) / PAGE;
        const long long v = (long long)npx * p.Hkv;
        if (v > 0 && lo < run + v) {
          bb = x; kk = (int)((lo - run) / npx); ll = (int)((lo - run) % npx); np = npx; hl = hx;
          break;
        }
        run += v;
      }
    }
    b0 = __shfl_sync(FULL, bb, src);
    kvh0 = __shfl_sync(FULL, kk, src);
    local0 = __shfl_sync(FULL, ll, src);
    np0 = __shfl_sync(FULL, np, src);
    hl0 = __shfl_sync(FULL, hl, src);
  }
}

}  // namespace split
}  // namespace oscar

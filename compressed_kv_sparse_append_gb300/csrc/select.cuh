// Block-wide exact top-K selection on order-preserving u32 keys.
//
// The top-K (largest keys; among equal keys the earliest elements) of n
// elements is found with an 8-bit radix select of the K-th largest key T
// (over the bits the keys do not all share), then an order-preserving
// compaction that keeps every key > T and the
// first `need` keys == T.  Elements are visited in array order, so when the
// array is in ascending entry order the output is the ascending index set and
// a tie at T goes to the lower entry index ("DeepSeek-V4 KV Cache 深度分析",
// §四: the indexer keeps the top-k blocks; equal scores resolved by index).
#pragma once

#include "common.cuh"

namespace ckv {

template <int NT>
struct SelectSmem {
  uint32_t hist[256];
  uint32_t warp_a[NT / 32];
  uint32_t warp_b[NT / 32];
  uint32_t bcast[4];
};

// Exclusive scan of (a, b) over the block; returns totals in ta, tb.
template <int NT>
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb,
                                            uint32_t& ta, uint32_t& tb, SelectSmem<NT>& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t xa = __shfl_up_sync(0xffffffffu, ia, o);
    uint32_t xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += xa;
      ib += xb;
    }
  }
  if (lane == 31) {
    sm.warp_a[warp] = ia;
    sm.warp_b[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t va = lane < NT / 32 ? sm.warp_a[lane] : 0u;
    uint32_t vb = lane < NT / 32 ? sm.warp_b[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t xa = __shfl_up_sync(0xffffffffu, va, o);
      uint32_t xb = __shfl_up_sync(0xffffffffu, vb, o);
      if (lane >= o) {
        va += xa;
        vb += xb;
      }
    }
    if (lane < NT / 32) {
      sm.warp_a[lane] = va;
      sm.warp_b[lane] = vb;
    }
  }
  __syncthreads();
  const uint32_t wa = warp ? sm.warp_a[warp - 1] : 0u, wb = warp ? sm.warp_b[warp - 1] : 0u;
  ea = wa + ia - a;
  eb = wb + ib - b;
  ta = sm.warp_a[NT / 32 - 1];
  tb = sm.warp_b[NT / 32 - 1];
  __syncthreads();
}

// Finds T (the K-th largest key among n, K <= n) and need = how many
// elements equal to T belong to the top-K.  get(i) returns element i's key.
// The bits every key shares (the common prefix of the smallest and largest
// key) are settled first; the rest is resolved 8 bits per pass, so scores of
// similar magnitude (which share their exponent bits) spread over the bins
// instead of piling onto one.
template <int NT, class Get>
__device__ void block_radix_threshold(int n, int K, Get get, SelectSmem<NT>& sm, uint32_t& T,
                                      uint32_t& need) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t u = get(i);
    lo = min(lo, u);
    hi = max(hi, u);
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    sm.warp_a[warp] = lo;
    sm.warp_b[warp] = hi;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t l2 = lane < NT / 32 ? sm.warp_a[lane] : 0xFFFFFFFFu;
    uint32_t h2 = lane < NT / 32 ? sm.warp_b[lane] : 0u;
    l2 = __reduce_min_sync(0xffffffffu, l2);
    h2 = __reduce_max_sync(0xffffffffu, h2);
    if (lane == 0) {
      sm.bcast[2] = l2;
      sm.bcast[3] = h2;
    }
  }
  __syncthreads();
  lo = sm.bcast[2];
  hi = sm.bcast[3];
  // (no barrier here: bcast[2..3] and warp_a/b are not written again before
  // the barriers below)
  if (lo == hi) {   // every key equal
    T = lo;
    need = (uint32_t)K;
    return;
  }
  int top = 32 - __clz(lo ^ hi);   // bits [top, 32) are the same in every key
  uint32_t prefix = top == 32 ? 0u : (lo & (0xFFFFFFFFu << top)), remaining = (uint32_t)K;
  // Two barriers per pass: warp 0 clears the bins as it scans them, and the
  // digit it publishes is read before any thread can reach the next pass's
  // publication (which follows that pass's first barrier).
  for (int i = threadIdx.x; i < 256; i += NT) sm.hist[i] = 0;
  __syncthreads();
#pragma unroll 1
  while (top > 0) {
    const int width = top < 8 ? top : 8, shift = top - width;
    const uint32_t mask = top == 32 ? 0u : (0xFFFFFFFFu << top);   // settled bits
    const uint32_t dmask = (1u << width) - 1u;
    for (int i = threadIdx.x; i < n; i += NT) {
      const uint32_t u = get(i);
      if (((u ^ prefix) & mask) == 0) atomicAdd(&sm.hist[(u >> shift) & dmask], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds digits 255-8l .. 248-8l (descending)
      uint32_t c[8], t = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sm.hist[255 - 8 * lane - j];
        sm.hist[255 - 8 * lane - j] = 0;
        t += c[j];
      }
      uint32_t incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      const uint32_t before = incl - t;
      const bool here = before < remaining && incl >= remaining;
      if (here) {
        uint32_t cum = before;
        for (int j = 0; j < 8; ++j) {
          if (cum + c[j] >= remaining) {
            sm.bcast[0] = (uint32_t)(255 - 8 * lane - j);
            sm.bcast[1] = remaining - cum;
            break;
          }
          cum += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= sm.bcast[0] << shift;
    remaining = sm.bcast[1];
    top = shift;
  }
  // the caller may reuse sm once everyone has read the last digit
  __syncthreads();
  T = prefix;
  need = remaining;
}

// Writes the top-K of n elements (or all n if n <= K) in array order via
// emit(out_pos, i).  Returns the number emitted.
template <int NT, class Get, class Emit>
__device__ int block_select_ordered(int n, int K, Get get, Emit emit, SelectSmem<NT>& sm,
                                    long long* marks = nullptr) {
  if (n <= 0 || K <= 0) return 0;
  const bool all = n <= K;
  uint32_t T = 0, need = 0;
  if (!all) block_radix_threshold<NT>(n, K, get, sm, T, need);
  if (marks && threadIdx.x == 0) marks[0] = clock64();
  const int per = (n + NT - 1) / NT;
  const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
  uint32_t gt = 0, eq = 0;
  if (!all) {
    for (int i = i0; i < i1; ++i) {
      const uint32_t u = get(i);
      gt += u > T;
      eq += u == T;
    }
  } else {
    gt = (uint32_t)(i1 - i0);
  }
  uint32_t gt_before, eq_before, gt_tot, eq_tot;
  block_scan2<NT>(gt, eq, gt_before, eq_before, gt_tot, eq_tot, sm);
  if (marks && threadIdx.x == 0) marks[1] = clock64();
  uint32_t pos = gt_before + min(eq_before, need);
  uint32_t eq_rank = eq_before;
  for (int i = i0; i < i1; ++i) {
    bool take = all;
    if (!all) {
      const uint32_t u = get(i);
      if (u > T) take = true;
      else if (u == T && eq_rank < need) {
        take = true;
        ++eq_rank;
      }
    }
    if (take) emit((int)pos++, i);
  }
  __syncthreads();
  return all ? n : K;
}

}  // namespace ckv

// Block-wide exact top-K selection on order-preserving u32 keys.
//
// The top-K (largest keys; among equal keys the earliest elements) of n
// elements is found with a radix select of the K-th largest key T (8 bits per
// pass over the bits the candidate keys do not all share), then an
// order-preserving compaction that keeps every key > T and the first `need`
// keys == T.  Elements are visited in array order, so when the array is in
// ascending entry order the output is the ascending index set and a tie at T
// goes to the lower entry index ("DeepSeek-V4 KV Cache 深度分析", §四: the
// indexer keeps the top-k blocks; equal scores resolved by index).
//
// This code runs once per CTA (the chunk's candidates) or once per sequence
// (the merge), so it executes with a cold instruction cache: it takes its keys
// from a run-time source and its loops handle one element per iteration, so
// that little code has to be fetched (unrolling them for more loads in flight
// made the merge slower: its time is mostly barriers and code fetch).
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

// Where the elements of a selection come from: element i's key and entry.
//   key != null: key[i] (shared memory); entry ent[i], or, with ent == null,
//                pool[i] (pool != null) or first + i.
//   key == null: the merge's candidate lists in global memory, element i
//                being slot i of their concatenation in chunk order (chunk c
//                holds slots cprefix[c] .. cprefix[c + 1] - 1, stored from
//                c * stride on).
struct SelSrc {
  const uint32_t* key;
  const int32_t* ent;
  const int32_t* pool;
  int64_t first;
  const uint32_t* gk;
  const int32_t* gi;
  const uint32_t* cprefix;
  int n_chunks;
  int64_t stride;

  __device__ int64_t slot(int v) const {
    int lo = 0, hi = n_chunks;   // last c with cprefix[c] <= v
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((int)cprefix[mid] <= v) lo = mid;
      else hi = mid;
    }
    return (int64_t)lo * stride + (v - (int)cprefix[lo]);
  }
  __device__ uint32_t k(int i) const { return key ? key[i] : __ldcg(gk + slot(i)); }
  __device__ int32_t e(int i) const {
    if (key) return ent ? ent[i] : pool ? pool[i] : (int32_t)(first + i);
    return __ldcg(gi + slot(i));
  }
};

// Finds T (the K-th largest key among n, K <= n) and need = how many
// elements equal to T belong to the top-K.  The bits every key shares (the
// common prefix of the smallest and largest key) are settled first; the rest
// is resolved 8 bits per pass.
//
// Hint: when the caller already knows that the K-th largest key has its top
// (32 - top0) bits equal to those of prefix0, and that `above` keys are
// larger than every key with that prefix, it passes top0 < 32, prefix0 and
// K - above as K: only the keys with that prefix take part.
template <int NT>
__device__ __forceinline__ void block_radix_threshold(const SelSrc src, int n, int K, SelectSmem<NT>& sm, uint32_t& T,
                                      uint32_t& need, uint32_t prefix0, int top0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t mask0 = top0 >= 32 ? 0u : (0xFFFFFFFFu << top0);
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll 1
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t u = src.k(i);
    if (((u ^ prefix0) & mask0) == 0u) {
      lo = min(lo, u);
      hi = max(hi, u);
    }
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
    // plain shared atomics (warp-aggregating them with match.any measured
    // far slower)
#pragma unroll 1
    for (int i = threadIdx.x; i < n; i += NT) {
      const uint32_t u = src.k(i);
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
#pragma unroll 1
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

// Writes the top-K of the n elements of `src` (or all n if n <= K) in array
// order: output position p receives the element's entry in out_ent[p] and,
// when out_key is not null, its key in out_key[p].  Hint (prefix0, top0,
// above) as for block_radix_threshold (top0 = 32: none).  Returns the number
// written.  Block-wide.
template <int NT>
__device__ __forceinline__ int select_ordered(const SelSrc src, int n, int K, uint32_t prefix0, int top0,
                                           int above, int32_t* out_ent, uint32_t* out_key,
                                           SelectSmem<NT>& sm) {
  if (n <= 0 || K <= 0) return 0;
  const bool all = n <= K;
  uint32_t T = 0, need = 0;
  if (!all) block_radix_threshold<NT>(src, n, K - above, sm, T, need, prefix0, top0);
  const int per = (n + NT - 1) / NT;
  const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
  uint32_t gt = 0, eq = 0;
  if (!all) {
#pragma unroll 1
    for (int i = i0; i < i1; ++i) {
      const uint32_t u = src.k(i);
      gt += u > T;
      eq += u == T;
    }
  } else {
    gt = (uint32_t)(i1 - i0);
  }
  uint32_t gt_before, eq_before, gt_tot, eq_tot;
  block_scan2<NT>(gt, eq, gt_before, eq_before, gt_tot, eq_tot, sm);
  uint32_t pos = gt_before + min(eq_before, need);
  uint32_t eq_rank = eq_before;
#pragma unroll 1
  for (int i = i0; i < i1; ++i) {
    bool take = all;
    uint32_t u = 0;
    if (!all || out_key) u = src.k(i);
    if (!all) {
      if (u > T) take = true;
      else if (u == T && eq_rank < need) {
        take = true;
        ++eq_rank;
      }
    }
    if (take) {
      out_ent[pos] = src.e(i);
      if (out_key) out_key[pos] = u;
      ++pos;
    }
  }
  __syncthreads();
  return all ? n : K;
}

}  // namespace ckv

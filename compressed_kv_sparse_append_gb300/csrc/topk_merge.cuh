// Candidate stage of csa_index_topk shared by the scorers.
//
// Each CTA keeps its chunk's top-K candidates (K = max(topk, pool_out)) in
// ascending entry order in the workspace and adds them to a per-sequence
// histogram of the top 12 key bits (global atomics).  The last CTA of the
// sequence (atomic ticket, no spinning) then
//   (a) finds the histogram bin holding the K-th largest key (and, when the
//       candidates in or above it would not fit in shared memory, the bin of
//       the next 12 key bits within it, from a second histogram over that
//       bin's candidates),
//   (b) compacts, in order, the candidates at or above that threshold into
//       shared memory (one pass over the candidate lists),
//   (c) runs the exact radix select on those survivors,
// and writes the ascending top-k (and the CSA2 Full layer's pool).  Ties at
// the threshold go to the earliest, i.e. lowest, entries ("DeepSeek-V4 KV
// Cache 深度分析", §四: the indexer keeps the top-k blocks).  If even that is
// too crowded for shared memory the select runs on the full lists.
#pragma once

#include "select.cuh"
#include "indexer.cuh"

namespace ckv {

constexpr int kHistShift = 20;                 // 12-bit histogram of the key
constexpr int kHistBins = 1 << (32 - kHistShift);

template <int NT>
struct MergeSmem {
  uint32_t pool_key[kMaxPool];
  int32_t pool_ent[kMaxPool];
  SelectSmem<NT> sel;
  int ticket;
  uint32_t n_real;
  uint32_t bcast[2];
};

// Final outputs from an ordered candidate source of n elements.
template <int NT, class GK, class GE>
__device__ void emit_outputs(const IndexArgs& a, int b, int n, int n_real, GK gk, GE ge,
                             MergeSmem<NT>& sm) {
  int32_t* oi = a.out_idx + (int64_t)b * a.topk;
  if (a.pool_out > 0) {
    const int kp = min(a.pool_out, n_real);
    block_select_ordered<NT>(
        n, kp, gk,
        [&](int pos, int i) {
          sm.pool_key[pos] = gk(i);
          sm.pool_ent[pos] = ge(i);
        },
        sm.sel);
    int32_t* op = a.out_pool + (int64_t)b * a.pool_out;
    for (int i = threadIdx.x; i < a.pool_out; i += NT) op[i] = i < kp ? sm.pool_ent[i] : -1;
    const int kk = min(a.topk, kp);
    block_select_ordered<NT>(
        kp, kk, [&](int i) { return sm.pool_key[i]; },
        [&](int pos, int i) { oi[pos] = sm.pool_ent[i]; }, sm.sel);
    for (int i = kk + threadIdx.x; i < a.topk; i += NT) oi[i] = -1;
  } else {
    const int kk = min(a.topk, n_real);
    block_select_ordered<NT>(n, kk, gk, [&](int pos, int i) { oi[pos] = ge(i); }, sm.sel);
    for (int i = kk + threadIdx.x; i < a.topk; i += NT) oi[i] = -1;
  }
}

// Of the kHistBins counts in hs (the last bin is the highest), finds the
// bin holding the min(K, total)-th largest element.  Returns the bin; sets
// total (all counts), keff = min(K, total) and above (the count in higher
// bins).  Block-wide; hs is only read.
template <int NT>
__device__ uint32_t find_bin_desc(const uint32_t* hs, uint32_t K, MergeSmem<NT>& sm, uint32_t& total,
                                  uint32_t& keff, uint32_t& above) {
  constexpr int per = (kHistBins + NT - 1) / NT;   // descending bins, contiguous per thread
  const int p0 = min(kHistBins, (int)threadIdx.x * per), p1 = min(kHistBins, p0 + per);
  uint32_t cnt = 0;
  for (int p = p0; p < p1; ++p) cnt += hs[kHistBins - 1 - p];
  uint32_t before, d0, d1;
  block_scan2<NT>(cnt, 0u, before, d0, total, d1, sm.sel);
  keff = min(K, total);
  if (threadIdx.x == 0) {
    sm.bcast[0] = 0u;
    sm.bcast[1] = 0u;
  }
  __syncthreads();
  if (keff > 0 && before < keff && before + cnt >= keff) {
    uint32_t cum = before;
    for (int p = p0; p < p1; ++p) {
      const uint32_t c = hs[kHistBins - 1 - p];
      if (cum + c >= keff) {
        sm.bcast[0] = (uint32_t)(kHistBins - 1 - p);
        sm.bcast[1] = cum;
        break;
      }
      cum += c;
    }
  }
  __syncthreads();
  const uint32_t bin = sm.bcast[0];
  above = sm.bcast[1];
  __syncthreads();
  return bin;
}

// Merge of all chunks' candidates (run by the last CTA of sequence b).
// surv_key / surv_ent: `surv_cap`-entry shared-memory scratch (>= kHistBins
// words for surv_key).  Every global read is a coalesced 16-byte load.
template <int NT>
__device__ void merge_and_emit(const IndexArgs& a, int b, MergeSmem<NT>& sm, uint32_t* surv_key,
                               int32_t* surv_ent, int surv_cap) {
  const bool tr = a.trace && b == 0 && threadIdx.x == 0;
  const long long t0 = clock64();
  const int n_slots = a.n_chunks * a.K_sel;   // K_sel is a multiple of 4
  const uint32_t* ck = a.cand_key + (int64_t)b * n_slots;
  const int32_t* ci = a.cand_idx + (int64_t)b * n_slots;
  uint32_t* hist = a.ghist + (int64_t)b * kHistBins;
  const int K = a.pool_out > 0 ? a.pool_out : a.topk;

  // (a) the histogram into shared memory (and zeroed for the next call)
  uint32_t* hs = surv_key;
  {
    // every load in flight before any store (the zeroing stores would
    // otherwise order each load after the previous one)
    constexpr int kV = kHistBins / 4, kPerT = (kV + NT - 1) / NT;
    uint4 hv[kPerT];
#pragma unroll
    for (int k = 0; k < kPerT; ++k) {
      const int v = threadIdx.x + k * NT;
      hv[k] = v < kV ? __ldcg(reinterpret_cast<const uint4*>(hist) + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kPerT; ++k) {
      const int v = threadIdx.x + k * NT;
      if (v < kV) {
        reinterpret_cast<uint4*>(hs)[v] = hv[k];
        reinterpret_cast<uint4*>(hist)[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  __syncthreads();
  uint32_t total, keff, above;
  const uint32_t tb = find_bin_desc<NT>(hs, (uint32_t)K, sm, total, keff, above);
  const int n_real = (int)total;
  // Survivors are the candidates with key >= lo_key.  When the threshold
  // bin is too crowded for shared memory (many exact ties at the boundary),
  // a second histogram of the next 12 key bits over that bin's candidates
  // narrows it first.
  uint32_t lo_key = tb << kHistShift;
  const uint32_t in_tb = hs[tb];
  if (keff > 0 && above + in_tb > (uint32_t)surv_cap) {
    __syncthreads();   // everyone has read hs[tb]
    for (int i = threadIdx.x; i < kHistBins; i += NT) hs[i] = 0u;
    __syncthreads();
    constexpr int kV2 = 4;   // 16-byte loads in flight per thread
    for (int base = 0; base < n_slots; base += 4 * kV2 * NT) {
      uint4 k4[kV2];
#pragma unroll
      for (int v = 0; v < kV2; ++v) {
        const int sv = base + 4 * (threadIdx.x + v * NT);
        k4[v] = sv < n_slots ? __ldcg(reinterpret_cast<const uint4*>(ck + sv)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int v = 0; v < kV2; ++v) {
        const uint32_t kk[4] = {k4[v].x, k4[v].y, k4[v].z, k4[v].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (kk[e] != 0u && (kk[e] >> kHistShift) == tb) atomicAdd(&hs[(kk[e] >> 8) & 0xFFFu], 1u);
      }
    }
    __syncthreads();
    uint32_t total2, keff2, above2;
    const uint32_t tb2 = find_bin_desc<NT>(hs, keff - above, sm, total2, keff2, above2);
    lo_key |= tb2 << 8;
  }
  trace_at(a.st, tr, 20, t0);

  // (b) survivors (key >= lo_key) in slot order, 16 slots per thread per
  // pass; the next pass's loads are issued before this pass is compacted
  constexpr int kPer = 16;
  uint32_t n_surv = 0;
  uint4 nk[kPer / 4];
  int4 ni[kPer / 4];
  auto fetch = [&](int base) {
    const int s0 = base + kPer * (int)threadIdx.x;
#pragma unroll
    for (int v = 0; v < kPer / 4; ++v) {
      const int sv = s0 + 4 * v;
      nk[v] = make_uint4(0u, 0u, 0u, 0u);
      ni[v] = make_int4(-1, -1, -1, -1);
      if (sv < n_slots) {
        nk[v] = __ldcg(reinterpret_cast<const uint4*>(ck + sv));
        ni[v] = __ldcg(reinterpret_cast<const int4*>(ci + sv));
      }
    }
  };
  fetch(0);
  for (int base = 0; base < n_slots; base += kPer * NT) {
    uint32_t kk[kPer];
    int32_t ii[kPer];
#pragma unroll
    for (int v = 0; v < kPer / 4; ++v) {
      kk[4 * v] = nk[v].x; kk[4 * v + 1] = nk[v].y; kk[4 * v + 2] = nk[v].z; kk[4 * v + 3] = nk[v].w;
      ii[4 * v] = ni[v].x; ii[4 * v + 1] = ni[v].y; ii[4 * v + 2] = ni[v].z; ii[4 * v + 3] = ni[v].w;
    }
    if (base + kPer * NT < n_slots) fetch(base + kPer * NT);
    uint32_t f = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) f |= (uint32_t)((kk[e] != 0u) && (kk[e] >= lo_key)) << e;
    uint32_t pos, d0, tot, d1;
    block_scan2<NT>((uint32_t)__popc(f), 0u, pos, d0, tot, d1, sm.sel);
    if (n_surv + tot <= (uint32_t)surv_cap) {
      pos += n_surv;
#pragma unroll
      for (int e = 0; e < kPer; ++e)
        if ((f >> e) & 1u) {
          surv_key[pos] = kk[e];
          surv_ent[pos] = ii[e];
          ++pos;
        }
    }
    n_surv += tot;
  }
  __syncthreads();
  trace_at(a.st, tr, 21, t0);
  if (tr) a.st->pad[23] = (int32_t)n_surv;
  if (n_surv <= (uint32_t)surv_cap) {
    emit_outputs<NT>(
        a, b, (int)n_surv, n_real, [&](int i) { return surv_key[i]; },
        [&](int i) { return surv_ent[i]; }, sm);
  } else {
    // a crowded threshold bin: select on the full lists in global memory
    emit_outputs<NT>(
        a, b, n_slots, n_real, [&](int i) { return __ldcg(ck + i); },
        [&](int i) { return __ldcg(ci + i); }, sm);
  }
  trace_at(a.st, tr, 22, t0);
}

// Local top-K of a scored chunk -> workspace (+ histogram); then the ticket.
// `scratch` (2 * surv_cap words of shared memory, free once the chunk's own
// selection is done) may alias `keys`.
template <int NT>
__device__ void chunk_select_and_merge(const IndexArgs& a, int b, int chunk, int n_elem,
                                       int64_t first_entry, const uint32_t* keys, uint32_t* scratch,
                                       int surv_cap, MergeSmem<NT>& sm) {
  const int slot0 = (b * a.n_chunks + chunk) * a.K_sel;
  uint32_t* ck = a.cand_key + slot0;
  int32_t* ci = a.cand_idx + slot0;
  uint32_t* hist = a.ghist + (int64_t)b * kHistBins;
  const int kk = min(a.K_sel, (int)sm.n_real);
  const int32_t* pool = a.pool ? a.pool + (int64_t)b * a.pool_len + first_entry : nullptr;
  const bool tr = a.trace && b == 0 && chunk == 0 && threadIdx.x == 0;
  if (a.n_chunks == 1 && a.pool_out == 0) {
    // one chunk holds the whole sequence: its top-k is the answer
    int32_t* oi = a.out_idx + (int64_t)b * a.topk;
    const int kt = min(a.topk, (int)sm.n_real);
    block_select_ordered<NT>(
        n_elem, kt, [&](int i) { return keys[i]; },
        [&](int pos, int i) { oi[pos] = pool ? pool[i] : (int32_t)(first_entry + i); }, sm.sel);
    for (int i = kt + threadIdx.x; i < a.topk; i += NT) oi[i] = -1;
    pdl_launch_dependents();
    return;
  }
  const long long t0 = clock64();
  long long marks[2] = {0, 0};
  block_select_ordered<NT>(
      n_elem, kk, [&](int i) { return keys[i]; },
      [&](int pos, int i) {
        const uint32_t u = keys[i];
        ck[pos] = u;
        ci[pos] = pool ? pool[i] : (int32_t)(first_entry + i);
        sm.pool_key[pos] = u;   // free until the merge
      },
      sm.sel, tr ? marks : nullptr);
  if (tr) {
    a.st->pad[12] = (int32_t)(marks[0] - t0);
    a.st->pad[13] = (int32_t)(marks[1] - t0);
  }
  for (int i = kk + threadIdx.x; i < a.K_sel; i += NT) {
    ck[i] = 0u;
    ci[i] = -1;
  }
  __syncthreads();
  // The candidates' keys crowd into a few histogram bins: one global atomic
  // per distinct bin per warp instead of one per candidate.
  {
    const int lane = threadIdx.x & 31;
    const int k_round = (kk + 31) / 32 * 32;
    for (int i = threadIdx.x; i < k_round; i += NT) {
      const uint32_t bin = i < kk ? (sm.pool_key[i] >> kHistShift) : 0xFFFFFFFFu;
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin != 0xFFFFFFFFu && (__ffs(peers) - 1) == lane) atomicAdd(hist + bin, (uint32_t)__popc(peers));
    }
  }
  trace_at(a.st, tr, 10, t0);
  __threadfence();
  __syncthreads();
  trace_at(a.st, tr, 11, t0);
  pdl_launch_dependents();   // the next kernel may take the SMs this grid frees
  if (threadIdx.x == 0) sm.ticket = (int)atomicAdd(a.counters + b, 1u);
  __syncthreads();
  if (sm.ticket != a.n_chunks - 1) return;
  __threadfence();
  merge_and_emit<NT>(a, b, sm, scratch, reinterpret_cast<int32_t*>(scratch + surv_cap), surv_cap);
  if (threadIdx.x == 0) atomicExch(a.counters + b, 0u);
}

}  // namespace ckv

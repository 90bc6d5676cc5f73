// Candidate stage of csa_index_topk shared by the scorers: the chunk's local
// top-K goes to the workspace in ascending entry order; the last CTA of the
// sequence (atomic ticket, no spinning) merges all chunks' candidates into
// the exact top-K (and, for a CSA2 Full layer, the top-k of that pool).
#pragma once

#include "select.cuh"
#include "indexer.cuh"

namespace ckv {

template <int NT>
struct MergeSmem {
  uint32_t pool_key[kMaxPool];
  int32_t pool_ent[kMaxPool];
  SelectSmem<NT> sel;
  int ticket;
  uint32_t n_real;
};

// Candidate merge and outputs (run by the last CTA of sequence b).
template <int NT>
__device__ void merge_and_emit(const IndexArgs& a, int b, MergeSmem<NT>& sm) {
  const int n_slots = a.n_chunks * a.K_sel;
  const uint32_t* ck = a.cand_key + (int64_t)b * n_slots;
  const int32_t* ci = a.cand_idx + (int64_t)b * n_slots;
  if (threadIdx.x == 0) sm.n_real = 0;
  __syncthreads();
  uint32_t mine = 0;
  for (int i = threadIdx.x; i < n_slots; i += NT) mine += __ldcg(ck + i) != 0u;
  atomicAdd(&sm.n_real, mine);
  __syncthreads();
  const int n_real = (int)sm.n_real;
  auto get = [&](int i) { return __ldcg(ck + i); };
  if (a.pool_out > 0) {
    const int kp = min(a.pool_out, n_real);
    block_select_ordered<NT>(
        n_slots, kp, get,
        [&](int pos, int i) {
          sm.pool_key[pos] = __ldcg(ck + i);
          sm.pool_ent[pos] = __ldcg(ci + i);
        },
        sm.sel);
    int32_t* op = a.out_pool + (int64_t)b * a.pool_out;
    for (int i = threadIdx.x; i < a.pool_out; i += NT) op[i] = i < kp ? sm.pool_ent[i] : -1;
    const int kk = min(a.topk, kp);
    int32_t* oi = a.out_idx + (int64_t)b * a.topk;
    block_select_ordered<NT>(
        kp, kk, [&](int i) { return sm.pool_key[i]; },
        [&](int pos, int i) { oi[pos] = sm.pool_ent[i]; }, sm.sel);
    for (int i = kk + threadIdx.x; i < a.topk; i += NT) oi[i] = -1;
  } else {
    const int kk = min(a.topk, n_real);
    int32_t* oi = a.out_idx + (int64_t)b * a.topk;
    block_select_ordered<NT>(
        n_slots, kk, get, [&](int pos, int i) { oi[pos] = __ldcg(ci + i); }, sm.sel);
    for (int i = kk + threadIdx.x; i < a.topk; i += NT) oi[i] = -1;
  }
}

// Local top-K of a scored chunk -> workspace; then the ticket.
template <int NT>
__device__ void chunk_select_and_merge(const IndexArgs& a, int b, int chunk, int n_elem,
                                       int64_t first_entry, const uint32_t* keys, MergeSmem<NT>& sm) {
  const int slot0 = (b * a.n_chunks + chunk) * a.K_sel;
  uint32_t* ck = a.cand_key + slot0;
  int32_t* ci = a.cand_idx + slot0;
  const int kk = min(a.K_sel, (int)sm.n_real);
  const int32_t* pool = a.pool ? a.pool + (int64_t)b * a.pool_len + first_entry : nullptr;
  block_select_ordered<NT>(
      n_elem, kk, [&](int i) { return keys[i]; },
      [&](int pos, int i) {
        ck[pos] = keys[i];
        ci[pos] = pool ? pool[i] : (int32_t)(first_entry + i);
      },
      sm.sel);
  for (int i = kk + threadIdx.x; i < a.K_sel; i += NT) {
    ck[i] = 0u;
    ci[i] = -1;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sm.ticket = (int)atomicAdd(a.counters + b, 1u);
  __syncthreads();
  if (sm.ticket != a.n_chunks - 1) return;
  __threadfence();
  merge_and_emit(a, b, sm);
  if (threadIdx.x == 0) atomicExch(a.counters + b, 0u);
}

}  // namespace ckv

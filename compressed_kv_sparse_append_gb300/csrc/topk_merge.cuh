// Candidate stage and cross-chunk merge of csa_index_topk, shared by the
// scorers ("DeepSeek-V4 KV Cache 深度分析", §四: the indexer keeps the top-k
// compressed blocks of the whole context).
//
// Every CTA scores one chunk of a sequence and builds, in shared memory, a
// histogram of its keys' top kBinBits bits while it scores.  Then:
//   1. it adds that histogram to the sequence's histogram in the workspace;
//   2. it reads the sequence histogram back.  Whatever other chunks have
//      added by then, if at least K keys lie in bins >= v, the sequence's
//      K-th largest key lies in a bin >= v: the highest such v is a lower
//      bound on the threshold bin.  (Counts read while others still add are
//      each at most the final count, so the bound holds for any snapshot.)
//   3. it writes its keys in bins >= that bound, in entry order, as its
//      candidates, with their count;
//   4. it takes a ticket; the last CTA of the sequence merges: the complete
//      histogram gives the threshold bin T and the count above it; the
//      candidates in bins >= T are exactly the sequence's keys there (every
//      chunk's bound is <= T); all candidates are staged in shared memory in
//      entry order, the keys of bin T are counted by their next 8 bits, and
//      an exact select restricted to that sub-bin picks the top K (a CSA2
//      Full layer does this twice: for its pool, then for its top-k).
// Equal keys go to the earliest, i.e. lowest, entries.  When more survivors
// reach the merge than its shared memory holds (a huge exact tie at the
// boundary), the select runs on the candidate lists in global memory.
#pragma once

#include "select.cuh"
#include "indexer.cuh"

namespace ckv {

__device__ __forceinline__ uint32_t key_bin(uint32_t key) { return key >> kBinShift; }

template <int NT>
struct MergeSmem {
  SelectSmem<NT> sel;
  uint32_t cprefix[kMaxChunksPerSeq + 1];   // merge: candidate offsets of the chunks
  uint32_t sprefix[kMaxChunksPerSeq + 1];   // merge: 4-aligned staging offsets of the chunks
  uint32_t wcnt[NT / 32];                   // per-warp counts of an ordered compaction
  uint32_t wcnt2[NT / 32];                  // second per-warp counts (keys equal to the threshold)
  uint32_t sub[256];                        // merge: next 8 key bits within the threshold bin
  int ticket;
  uint32_t n_real;                          // real keys of this chunk
  uint32_t kmin, kmax;                      // smallest / largest real key of this chunk
  uint32_t bcast[4];
};

// Sets n_real / kmin / kmax before the scorer's keys are written.
template <int NT>
__device__ __forceinline__ void merge_smem_init(MergeSmem<NT>& sm) {
  if (threadIdx.x == 0) {
    sm.n_real = 0u;
    sm.kmin = 0xFFFFFFFFu;
    sm.kmax = 0u;
  }
}

// Descending scan of the histogram `gh` (global, read through L2) from bin
// top - 1 down: returns the highest bin v with (count of bins >= v) >= K, or
// 0 if the whole histogram holds fewer.  `above` = count in bins > v.
// Block-wide; NT bins per round, one load each.
template <int NT>
__device__ uint32_t hist_bin_from_top(const uint32_t* gh, int top, uint32_t K, MergeSmem<NT>& sm,
                                      uint32_t& above) {
  uint32_t carry = 0;
  for (int hi = top; hi > 0; hi -= NT) {
    const int bin = hi - 1 - (int)threadIdx.x;
    const uint32_t v = bin >= 0 ? __ldcg(gh + bin) : 0u;
    uint32_t before, tot, d0, d1;
    block_scan2<NT>(v, 0u, before, d0, tot, d1, sm.sel);
    if (threadIdx.x == 0) sm.bcast[0] = 0xFFFFFFFFu;
    __syncthreads();
    if (v > 0 && carry + before < K && carry + before + v >= K) {
      sm.bcast[0] = (uint32_t)bin;
      sm.bcast[1] = carry + before;
    }
    __syncthreads();
    const uint32_t found = sm.bcast[0];
    if (found != 0xFFFFFFFFu) {
      above = sm.bcast[1];
      __syncthreads();
      return found;
    }
    carry += tot;
  }
  above = carry;
  return 0u;
}

// The chunk's lower bound on its sequence's threshold bin: one descending
// scan from bin top - 1 over two histograms at once -- the sequence's (global,
// a snapshot while other chunks still add to it; this chunk's own additions
// may or may not be visible yet) and this chunk's own (shared memory).  The
// highest bin at which either reaches K keys from the top is a valid bound
// (each count is at most the sequence's true count).  0 if neither does.
template <int NT>
__device__ uint32_t chunk_bound(const uint32_t* gh, const uint32_t* lh, int top, uint32_t K,
                                MergeSmem<NT>& sm) {
  uint32_t cg = 0, cl = 0;
  uint32_t found_g = 0xFFFFFFFFu, found_l = 0xFFFFFFFFu;
  for (int hi = top; hi > 0; hi -= NT) {
    const int bin = hi - 1 - (int)threadIdx.x;
    const uint32_t vg = bin >= 0 ? __ldcg(gh + bin) : 0u;
    const uint32_t vl = bin >= 0 ? lh[bin] : 0u;
    uint32_t bg, bl, tg, tl;
    block_scan2<NT>(vg, vl, bg, bl, tg, tl, sm.sel);
    if (threadIdx.x == 0) {
      sm.bcast[0] = 0xFFFFFFFFu;
      sm.bcast[1] = 0xFFFFFFFFu;
    }
    __syncthreads();
    if (found_g == 0xFFFFFFFFu && vg > 0 && cg + bg < K && cg + bg + vg >= K) sm.bcast[0] = (uint32_t)bin;
    if (found_l == 0xFFFFFFFFu && vl > 0 && cl + bl < K && cl + bl + vl >= K) sm.bcast[1] = (uint32_t)bin;
    __syncthreads();
    if (sm.bcast[0] != 0xFFFFFFFFu) found_g = sm.bcast[0];
    if (sm.bcast[1] != 0xFFFFFFFFu) found_l = sm.bcast[1];
    cg += tg;
    cl += tl;
    __syncthreads();
    // the local bound is never above the global one once both are found;
    // either alone already bounds, and the scan stops at the first found
    if (found_g != 0xFFFFFFFFu || found_l != 0xFFFFFFFFu) break;
  }
  const uint32_t g = found_g == 0xFFFFFFFFu ? 0u : found_g;
  const uint32_t l = found_l == 0xFFFFFFFFu ? 0u : found_l;
  return g > l ? g : l;
}

// Final outputs from an ordered source of n elements (n_real real keys in
// the sequence).  Hint (prefix0, top0, above): the K-th largest key has
// prefix0's top (32 - top0) bits and `above` keys lie above all such keys
// (top0 = 32: none).  With `pooled`, a CSA2 Full layer's pool is written
// first (key and entry also kept in shared memory) and the top-k is then
// taken from the pool: two selections run through one call site.
template <int NT>
__device__ void emit_outputs(const IndexArgs& a, int b, SelSrc src, int n, int n_real,
                             uint32_t* pool_key, int32_t* pool_ent, MergeSmem<NT>& sm,
                             uint32_t prefix0, int top0, int above, bool pooled) {
  int32_t* oi = a.out_idx + (int64_t)b * a.topk;
  int kk = min(a.topk, n_real);
  int K = pooled ? min(a.pool_out, n_real) : kk;
#pragma unroll 1
  for (int job = 0; job < (pooled ? 2 : 1); ++job) {
    const bool to_pool = pooled && job == 0;
    select_ordered<NT>(src, n, K, prefix0, top0, above, to_pool ? pool_ent : oi,
                       to_pool ? pool_key : nullptr, sm.sel);
    if (to_pool) {
      int32_t* op = a.out_pool + (int64_t)b * a.pool_out;
#pragma unroll 1
      for (int i = threadIdx.x; i < a.pool_out; i += NT) op[i] = i < K ? pool_ent[i] : -1;
      // second job: the top-k of the pool, no hint
      src = SelSrc{};
      src.key = pool_key;
      src.ent = pool_ent;
      n = K;
      kk = min(a.topk, K);
      K = kk;
      prefix0 = 0u;
      top0 = 32;
      above = 0;
    }
  }
#pragma unroll 1
  for (int i = kk + threadIdx.x; i < a.topk; i += NT) oi[i] = -1;
}

// Writes, in array order, every element of key[0, n) above T and the first
// `need` equal to T (the top-K once T and need are those of its K-th largest
// key): output position = (keys > T before it) + min(keys == T before it,
// need).  Rounds of NT x 8 elements, each lane's eight in flight; one ballot
// pair per 32 elements and one barrier per round.  Block-wide.
template <int NT>
__device__ __forceinline__ void emit_ordered(const uint32_t* key, const int32_t* ent, int n, uint32_t T,
                                             uint32_t need, int32_t* out, MergeSmem<NT>& sm) {
  constexpr int kU = 8, kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t g_run = 0, e_run = 0;   // keys > T and == T in earlier rounds
#pragma unroll 1
  for (int base = 0; base < n; base += NT * kU) {
    const int wbase = base + warp * 32 * kU;
    uint32_t bg[kU], be[kU], cg = 0, ce = 0;
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int v = wbase + k * 32 + lane;
      const uint32_t u = v < n ? key[v] : 0u;
      bg[k] = __ballot_sync(0xffffffffu, u > T);
      be[k] = __ballot_sync(0xffffffffu, u == T && u != 0u);
      cg += __popc(bg[k]);
      ce += __popc(be[k]);
    }
    if (lane == 0) {
      sm.wcnt[warp] = cg;
      sm.wcnt2[warp] = ce;
    }
    __syncthreads();
    // every warp scans the warps' counts: its exclusive prefix and the totals
    const uint32_t xg = lane < kWarps ? sm.wcnt[lane] : 0u, xe = lane < kWarps ? sm.wcnt2[lane] : 0u;
    uint32_t ig = xg, ie = xe;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t yg = __shfl_up_sync(0xffffffffu, ig, o), ye = __shfl_up_sync(0xffffffffu, ie, o);
      if (lane >= o) {
        ig += yg;
        ie += ye;
      }
    }
    uint32_t g = g_run + __shfl_sync(0xffffffffu, ig - xg, warp);
    uint32_t e = e_run + __shfl_sync(0xffffffffu, ie - xe, warp);
    g_run += __shfl_sync(0xffffffffu, ig, kWarps - 1);
    e_run += __shfl_sync(0xffffffffu, ie, kWarps - 1);
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int v = wbase + k * 32 + lane;
      const uint32_t gb = g + __popc(bg[k] & lt), eb = e + __popc(be[k] & lt);
      if ((bg[k] >> lane) & 1u) out[gb + min(eb, need)] = ent[v];
      else if (((be[k] >> lane) & 1u) && eb < need) out[gb + eb] = ent[v];
      g += __popc(bg[k]);
      e += __popc(be[k]);
    }
    __syncthreads();   // wcnt is written again by the next round
  }
}

// The staged candidates whose top bits equal `prefix` (under hmask) into
// the list (key, staged position; list slots past 2 x NT are dropped, the
// count in sm.bcast[2] still counts them); with BM, every bitmap word of
// bmA covered (32 consecutive candidates, from a warp's ballot) marks the
// keys above that prefix and the same word of bmE is cleared.  Eight keys
// per lane in flight, one counter update per warp and round.  Block-wide;
// sm.bcast[2] must be 0 on entry (barrier after).
template <int NT, bool BM>
__device__ __forceinline__ void gather_sub_bin(const uint32_t* surv_key, int n_pad, uint32_t hmask,
                                               uint32_t prefix, uint32_t* lkey, uint32_t* lpos,
                                               uint32_t* bmA, uint32_t* bmE, MergeSmem<NT>& sm) {
  constexpr int kU = 8, kListMax = 2 * NT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll 1
  for (int w0 = warp * 32 * kU; w0 < n_pad; w0 += NT * kU) {
    uint32_t u[kU], bal[kU], c = 0;
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int i = w0 + k * 32 + lane;
      u[k] = i < n_pad ? surv_key[i] : 0u;
      bal[k] = __ballot_sync(0xffffffffu, u[k] != 0u && (u[k] & hmask) == prefix);
      if (BM) {
        const uint32_t ba = __ballot_sync(0xffffffffu, (u[k] & hmask) > prefix);
        if (lane == 0) {
          bmA[(w0 >> 5) + k] = ba;
          bmE[(w0 >> 5) + k] = 0u;
        }
      }
      c += __popc(bal[k]);
    }
    if (c == 0u) continue;   // warp-uniform
    uint32_t at = 0u;
    if (lane == 0) at = atomicAdd(&sm.bcast[2], c);
    at = __shfl_sync(0xffffffffu, at, 0);
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const uint32_t x = at + __popc(bal[k] & lt);
      if (((bal[k] >> lane) & 1u) && x < (uint32_t)kListMax) {
        lkey[x] = u[k];
        lpos[x] = (uint32_t)(w0 + k * 32 + lane);
      }
      at += __popc(bal[k]);
    }
  }
}

// Leaves the sequence's histogram (bins in use: below seq[1] = top, from
// kBins - seq[2] up) and its state words zero for the next call.  Block-wide.
template <int NT>
__device__ __forceinline__ void clear_sequence_state(uint32_t* gh, uint32_t* seq, int top) {
  const int bot = kBins - (int)__ldcg(seq + 2);
  if (top > 0) {
    const int z0 = bot & ~3, z1 = (top + 3) & ~3;
    for (int v = z0 / 4 + (int)threadIdx.x; v < z1 / 4; v += NT)
      reinterpret_cast<uint4*>(gh)[v] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();   // every thread has read seq[2] before it is cleared
  if (threadIdx.x == 0) {
    seq[1] = 0u;
    seq[2] = 0u;
    seq[0] = 0u;
  }
}

// Merge of the sequence's candidates, run by its last CTA.  `scratch`
// (scratch_words 32-bit words of shared memory, dead otherwise) holds the
// survivors and, for a CSA2 Full layer, the pool.  BM: the kernel instance
// for long sequences, whose merge writes the output of a large staged set
// from bitmaps (the code stays out of the other instance).
template <int NT, bool BM>
__device__ void merge_and_emit(const IndexArgs& a, int b, MergeSmem<NT>& sm, uint32_t* scratch,
                               int scratch_words, uint32_t own_bound) {
  const bool tr = a.trace && b == 0 && threadIdx.x == 0;
  const long long t0 = clock64();
  const int K = a.pool_out > 0 ? a.pool_out : a.topk;
  const int nch = a.n_chunks;
  uint32_t* seq = a.seq_state + (int64_t)b * kSeqWords;
  uint32_t* gh = a.ghist + (int64_t)b * kBins;
  const uint2* cc = reinterpret_cast<const uint2*>(a.ccount) + (int64_t)b * nch;

  // One round trip for: the chunks' counts, the top bin in use, and the
  // histogram window [own_bound, own_bound + NT) (this CTA's bound is a
  // lower bound on the threshold bin, so when no key lies above the window
  // the window alone gives the threshold bin).
  const int wbin = (int)own_bound + (int)threadIdx.x;
  const uint32_t wv = (own_bound > 0 && wbin < kBins) ? __ldcg(gh + wbin) : 0u;
  const int top = (int)__ldcg(seq + 1);
  // chunk candidate counts -> offsets; real keys in total
  uint32_t n_total = 0;
  {
    constexpr int kPer = (kMaxChunksPerSeq + NT - 1) / NT;
    const int c0 = min(nch, (int)threadIdx.x * kPer), c1 = min(nch, c0 + kPer);
    uint32_t cnt[kPer], real = 0, mine = 0, mine4 = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      cnt[k] = 0u;
      if (c0 + k < c1) {
        const uint2 v = __ldcg(cc + c0 + k);
        cnt[k] = v.x;
        real += v.y;
        mine += v.x;
        mine4 += (v.x + 3u) & ~3u;
      }
    }
    uint32_t before, before4, tot, tot4, d0, rt;
    block_scan2<NT>(mine, mine4, before, before4, tot, tot4, sm.sel);
    block_scan2<NT>(real, 0u, d0, d0, rt, d0, sm.sel);
    n_total = rt;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (c0 + k < c1) {
        sm.cprefix[c0 + k] = before;
        sm.sprefix[c0 + k] = before4;
        before += cnt[k];
        before4 += (cnt[k] + 3u) & ~3u;
      }
    if (threadIdx.x == 0) {
      sm.cprefix[nch] = tot;
      sm.sprefix[nch] = tot4;
    }
    __syncthreads();
  }
  const int n_cand = (int)sm.cprefix[nch];
  const int n_pad = (int)sm.sprefix[nch];   // staged length: chunk lists padded to 4 entries
  const int keff = min(K, (int)n_total);
  constexpr int kWarps = NT / 32;
  const int pool_words = a.pool_out > 0 ? 2 * kMaxPool : 0;
  const int surv_cap = ((scratch_words - pool_words - kWarps * 256) / 2) & ~3;
  const bool pooled = a.pool_out > 0;
  // Every key is a survivor when the sequence has at most K.  Otherwise the
  // K-th largest key is located by its bin in the complete sequence
  // histogram (the threshold bin), then by the next 8 bits of the
  // candidates in that bin (the sub-bin); an exact select among the keys of
  // that sub-bin alone decides it.
  const bool hint = keff > 0 && (int)n_total > K;
  // Threshold bin of the kk-th largest key and the count of keys in the bins
  // above it: from the window read with the counts when that window reaches
  // the top bin in use (this CTA's bound is a lower bound on the threshold
  // bin of any kk <= K), else by a scan from the top.
  auto threshold_bin = [&](uint32_t kk, uint32_t& tb_, uint32_t& above_) {
    bool done = false;
    if (own_bound > 0 && top <= (int)own_bound + NT) {
      uint32_t before, d0, tot, d1;
      block_scan2<NT>(wv, 0u, before, d0, tot, d1, sm.sel);
      if (threadIdx.x == 0) sm.bcast[0] = 0xFFFFFFFFu;
      __syncthreads();
      const uint32_t hi_cnt = tot - before - wv;   // keys in window bins above this one
      if (wv > 0 && hi_cnt < kk && hi_cnt + wv >= kk) {
        sm.bcast[0] = (uint32_t)wbin;
        sm.bcast[1] = hi_cnt;
      }
      __syncthreads();
      if (sm.bcast[0] != 0xFFFFFFFFu) {
        tb_ = sm.bcast[0];
        above_ = sm.bcast[1];
        done = true;
      }
      __syncthreads();
    }
    if (!done) tb_ = hist_bin_from_top<NT>(gh, top, kk, sm, above_);
    __syncthreads();   // every thread has read bcast before it is written again
  };

  // Every candidate into shared memory, in entry order (chunk c's list at
  // offset sprefix[c], padded to a multiple of 4 entries whose padding keys
  // are 0, i.e. no key): one warp per chunk list, 16-byte asynchronous
  // copies, all of them in flight while the threshold bin is found.
  uint32_t* surv_key = scratch;
  int32_t* surv_ent = reinterpret_cast<int32_t*>(scratch + surv_cap);
  uint32_t* wsub = scratch + 2 * surv_cap;            // [warp][256] private sub-bin counts
  uint32_t* pool_key = wsub + kWarps * 256;
  int32_t* pool_ent = reinterpret_cast<int32_t*>(pool_key + kMaxPool);
  SelSrc cl{};   // the candidate lists in global memory
  cl.gk = a.cand_key + (int64_t)b * nch * a.chunk;
  cl.gi = a.cand_idx + (int64_t)b * nch * a.chunk;
  cl.cprefix = sm.cprefix;
  cl.n_chunks = nch;
  cl.stride = a.chunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kWarps * 256; i += NT) wsub[i] = 0u;
  const bool staged = n_pad <= surv_cap;
  if (staged) {
    // (the chunk lists start 16-byte aligned in global memory: a.chunk is a
    // multiple of 4; reading up to 3 slots past a list stays in its chunk,
    // and those slots hold whatever an earlier call left there)
#pragma unroll 1
    for (int c = warp; c < nch; c += kWarps) {
      const int cnt = (int)(sm.cprefix[c + 1] - sm.cprefix[c]);
      const int groups = (cnt + 3) >> 2;
      const uint32_t* gk = cl.gk + (int64_t)c * a.chunk;
      const int32_t* gi = cl.gi + (int64_t)c * a.chunk;
      const uint32_t dk = smem_u32(surv_key + sm.sprefix[c]), de = smem_u32(surv_ent + sm.sprefix[c]);
#pragma unroll 1
      for (int g = lane; g < groups; g += 32) {
        cp_async16(dk + 16 * g, gk + 4 * g);
        cp_async16(de + 16 * g, gi + 4 * g);
      }
    }
  }
  uint32_t tb = 0, above = 0;
  if (hint) threshold_bin((uint32_t)keff, tb, above);
  const uint32_t lo_key = tb << kBinShift;
  trace_at(a.st, tr, 20, t0);
  if (staged) {
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();   // every copy has landed
    // the padding slots of every list become "no key"
    for (int c = threadIdx.x; c < nch; c += NT) {
      const int cnt = (int)(sm.cprefix[c + 1] - sm.cprefix[c]);
      for (int k = cnt; k < ((cnt + 3) & ~3); ++k) surv_key[sm.sprefix[c] + k] = 0u;
    }
  }
  __syncthreads();
  uint32_t n_surv = (uint32_t)n_pad;
  if (tr) a.st->pad[17] = (int32_t)(clock64() - t0);
  if (tr) {
    a.st->pad[23] = (int32_t)n_surv;
    a.st->pad[25] = n_cand;
    a.st->pad[26] = (int32_t)tb;
    a.st->pad[27] = (int32_t)above;
    a.st->pad[28] = (int32_t)n_total;
  }
  bool pool_left = pooled;   // the pool is still to be written
  uint32_t prefix = lo_key, above2 = above;
  int top_bits = kBinShift;
  if (hint && staged) {
    // One job per output: the top-K (for a pool-building call, the pool,
    // then the top-k of the pool, which is the top-k of the sequence).  Per
    // job: the keys of the threshold bin counted by their next 8 bits, the
    // sub-bin holding the job's K-th largest, its keys (with their staged
    // positions) gathered into a list in the dead sub-bin counters, the
    // threshold T and the count `need` of keys equal to T to keep found on
    // the list alone (every key above the sub-bin is kept), then the output
    // written by one ordered pass over the staged candidates or, in the
    // long-sequence instance with many staged, from bitmaps.
    constexpr int kListMax = 2 * NT;   // 2 x kListMax words fit in wsub
    constexpr int kRankMax = 64;
    uint32_t* lkey = wsub;
    uint32_t* lpos = wsub + kListMax;
    int32_t* oi = a.out_idx + (int64_t)b * a.topk;
#pragma unroll 1
    for (int job = 0;; ++job) {
      const uint32_t kj = job == 0 ? (uint32_t)keff : (uint32_t)min(a.topk, keff);
      if (job > 0) {
        threshold_bin(kj, tb, above);
        for (int i = threadIdx.x; i < kWarps * 256; i += NT) wsub[i] = 0u;   // the list's words
        __syncthreads();
      }
      if (threadIdx.x == 0) {
        sm.bcast[0] = 0u;   // sub-bin search defaults
        sm.bcast[1] = 0u;
      }
      {
        // warp-private counters (no contention between warps on the few
        // sub-bins that exact ties crowd), four independent elements per
        // lane, plain shared atomics (match.any aggregation measured far
        // slower)
        uint32_t* ws = wsub + warp * 256;
#pragma unroll 1
        for (int i0 = threadIdx.x; i0 < n_pad; i0 += 4 * NT) {
          uint32_t u[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) u[k] = i0 + k * NT < n_pad ? surv_key[i0 + k * NT] : 0u;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (key_bin(u[k]) == tb && u[k] != 0u) atomicAdd(&ws[(u[k] >> (kBinShift - 8)) & 255u], 1u);
        }
        __syncthreads();
        for (int v = threadIdx.x; v < 256; v += NT) {
          uint32_t t = 0;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) t += wsub[w * 256 + v];
          sm.sub[v] = t;
        }
        __syncthreads();
      }
      trace_at(a.st, tr, 21, t0);
      {
        // the sub-bin of the threshold bin that holds the kj-th largest key
        const uint32_t need = kj - above;
        if (warp == 0) {
          // lane l holds sub-bins 255 - 8l .. 248 - 8l (descending)
          uint32_t c8[8], t8 = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            c8[j] = sm.sub[255 - 8 * lane - j];
            t8 += c8[j];
          }
          uint32_t incl = t8;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const uint32_t before = incl - t8;
          if (before < need && incl >= need) {
            uint32_t cum = before;
            for (int j = 0; j < 8; ++j) {
              if (cum + c8[j] >= need) {
                sm.bcast[0] = (uint32_t)(255 - 8 * lane - j);
                sm.bcast[1] = cum;
                break;
              }
              cum += c8[j];
            }
          }
        }
        __syncthreads();
        const uint32_t t2 = sm.bcast[0] & 255u;
        above2 = above + sm.bcast[1];
        prefix = (tb << kBinShift) | (t2 << (kBinShift - 8));
        top_bits = kBinShift - 8;
      }
      if (threadIdx.x == 0) sm.bcast[2] = 0u;
      __syncthreads();
      const uint32_t hmask = ~((1u << top_bits) - 1u);
      // Long-sequence instance, more staged candidates than one ordered pass
      // takes in a round: one bit per staged candidate, in words after the
      // list, where bmA marks the keys above the sub-bin (and later the
      // list's keys above T) and bmE the list's keys equal to T, and the
      // output is written from the bitmaps.  The gather below then writes
      // every word of bmA and bmE it covers (up to kU words past the staged
      // length).
      constexpr int kU = 8;
      const int n_words = (n_pad + 31) >> 5;
      uint32_t* bmA = lpos + kListMax;
      uint32_t* bmE = bmA + n_words + kU;
      const bool use_bm = BM && n_pad > NT * kU && 2 * kListMax + 2 * (n_words + kU) <= kWarps * 256;
      if (use_bm) gather_sub_bin<NT, true>(surv_key, n_pad, hmask, prefix, lkey, lpos, bmA, bmE, sm);
      else gather_sub_bin<NT, false>(surv_key, n_pad, hmask, prefix, lkey, lpos, bmA, bmE, sm);
      __syncthreads();
      const int m = (int)sm.bcast[2];
      if (m > kListMax) break;   // a crowded sub-bin: the compaction below
      const uint32_t need2 = kj - above2;   // in [1, m] by the sub-bin search
      uint32_t T = 0, need = 0;
      if (m <= kRankMax) {
        // rank of each list key: larger keys first, equal keys by position;
        // the key of rank need2 - 1 is T (m^2 comparisons: short lists only)
        if ((int)threadIdx.x < m) {
          const uint32_t u = lkey[threadIdx.x], ps = lpos[threadIdx.x];
          uint32_t r = 0, gt = 0;
          auto rank_one = [&](uint32_t uj, uint32_t pj) {
            gt += uj > u;
            r += uj > u || (uj == u && pj < ps);
          };
          // four list entries per 16-byte load (the list starts 16-byte
          // aligned), several loads in flight
          const int m4 = m & ~3;
#pragma unroll 4
          for (int j = 0; j < m4; j += 4) {
            const uint4 kq = *reinterpret_cast<const uint4*>(lkey + j);
            const uint4 pq = *reinterpret_cast<const uint4*>(lpos + j);
            rank_one(kq.x, pq.x);
            rank_one(kq.y, pq.y);
            rank_one(kq.z, pq.z);
            rank_one(kq.w, pq.w);
          }
#pragma unroll 1
          for (int j = m4; j < m; ++j) rank_one(lkey[j], lpos[j]);
          if (r == need2 - 1u) {
            sm.bcast[0] = u;
            sm.bcast[1] = need2 - gt;
          }
        }
        __syncthreads();
        T = sm.bcast[0];
        need = sm.bcast[1];
        __syncthreads();
      } else {
        SelSrc ls{};
        ls.key = lkey;
        block_radix_threshold<NT>(ls, m, (int)need2, sm.sel, T, need, prefix, top_bits);
      }
      trace_at(a.st, tr, 19, t0);
      if (tr) a.st->pad[31] = m;
      int32_t* out = pool_left ? a.out_pool + (int64_t)b * a.pool_out : oi;
      const int len = pool_left ? a.pool_out : a.topk;
      if (!use_bm) {
        emit_ordered<NT>(surv_key, surv_ent, n_pad, T, need, out, sm);
      } else {
        // the list's keys above T and equal to T into the bitmaps
#pragma unroll 1
        for (int i = threadIdx.x; i < m; i += NT) {
          const uint32_t u = lkey[i], ps = lpos[i];
          if (u > T) atomicOr(&bmA[ps >> 5], 1u << (ps & 31u));
          else if (u == T) atomicOr(&bmE[ps >> 5], 1u << (ps & 31u));
        }
        __syncthreads();
        // Output position of a kept candidate = keys above T before it +
        // min(keys equal to T before it, need), counted on the bitmaps:
        // each thread a contiguous run of words, one scan of their counts.
        const int per = (n_words + NT - 1) / NT;
        const int wlo = min(n_words, (int)threadIdx.x * per), whi = min(n_words, wlo + per);
        uint32_t ca = 0, ce = 0;
#pragma unroll 1
        for (int w = wlo; w < whi; ++w) {
          ca += __popc(bmA[w]);
          ce += __popc(bmE[w]);
        }
        uint32_t pa, pe, ta, te;
        block_scan2<NT>(ca, ce, pa, pe, ta, te, sm.sel);
#pragma unroll 1
        for (int w = wlo; w < whi; ++w) {
          const uint32_t wa = bmA[w], we = bmE[w];
          uint32_t x = wa | we;
          while (x) {
            const int bit = __ffs(x) - 1;
            x &= x - 1u;
            const uint32_t lo = (1u << bit) - 1u;
            const uint32_t na = pa + __popc(wa & lo), ne = pe + __popc(we & lo);
            const int32_t ent = surv_ent[w * 32 + bit];
            // (positions stay below kj by the choice of T and need; the
            // test keeps a write inside the output row regardless)
            if ((wa >> bit) & 1u) {
              const uint32_t at = na + min(ne, need);
              if (at < kj) out[at] = ent;
            } else if (ne < need && na + ne < kj) {
              out[na + ne] = ent;
            }
          }
          pa += __popc(wa);
          pe += __popc(we);
        }
      }
#pragma unroll 1
      for (int i = (int)kj + (int)threadIdx.x; i < len; i += NT) out[i] = -1;
      if (pool_left) {
        pool_left = false;
        continue;
      }
      trace_at(a.st, tr, 22, t0);
      clear_sequence_state<NT>(gh, seq, top);
      return;
    }
  }
  if (staged && (hint || n_pad != n_cand)) {
    // in-place ordered compaction to the real keys >= prefix (without a
    // hint prefix is 0: only the padding goes), kU per thread per round (a
    // round's reads all happen before its writes, which never reach past it)
    constexpr int kU = 8;
    uint32_t kept = 0;
#pragma unroll 1
    for (int base = 0; base < (int)n_surv; base += NT * kU) {
      const int wbase = base + warp * 32 * kU;
      uint32_t u[kU];
      int32_t x[kU];
      uint32_t bal[kU], cnt = 0;
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        const int v = wbase + k * 32 + lane;
        u[k] = v < (int)n_surv ? surv_key[v] : 0u;
        x[k] = v < (int)n_surv ? surv_ent[v] : -1;
      }
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        bal[k] = __ballot_sync(0xffffffffu, u[k] != 0u && u[k] >= prefix);
        cnt += __popc(bal[k]);
      }
      if (lane == 0) sm.wcnt[warp] = cnt;
      __syncthreads();
      uint32_t pos = kept, tot = 0;
#pragma unroll 1
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = sm.wcnt[w];
        pos += w < warp ? c : 0u;
        tot += c;
      }
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        if ((bal[k] >> lane) & 1u) {
          const uint32_t at = pos + __popc(bal[k] & ((1u << lane) - 1u));
          surv_key[at] = u[k];
          surv_ent[at] = x[k];
        }
        pos += __popc(bal[k]);
      }
      kept += tot;
      __syncthreads();
    }
    n_surv = kept;
  }
  trace_at(a.st, tr, 19, t0);
  if (tr) a.st->pad[31] = (int32_t)n_surv;
  if (staged) {
    SelSrc ss{};
    ss.key = surv_key;
    ss.ent = surv_ent;
    emit_outputs<NT>(a, b, ss, (int)n_surv, (int)n_total, pool_key, pool_ent, sm, prefix,
                     hint ? top_bits : 32, hint ? (int)above2 : 0, pool_left);
  } else {
    // a crowded threshold bin: select on the candidate lists in global memory
    emit_outputs<NT>(a, b, cl, n_cand, (int)n_total, pool_key, pool_ent, sm, lo_key,
                     hint ? kBinShift : 32, hint ? (int)above : 0, pool_left);
  }
  trace_at(a.st, tr, 22, t0);
  clear_sequence_state<NT>(gh, seq, top);
}

// After scoring: `keys[0, n_elem)` hold this chunk's keys (0 = no entry),
// `hist` (kBins words of shared memory) their histogram, sm.n_real / kmin /
// kmax the count and range of real keys.  Publishes the histogram, writes
// the chunk's candidates and takes the ticket; the last CTA merges.
// `scratch` (scratch_words words of shared memory, dead after this chunk's
// candidates are written; may alias `keys` and `hist`) serves the merge.
template <int NT, bool BM = false>
__device__ void chunk_select_and_merge(const IndexArgs& a, int b, int chunk, int n_elem,
                                       int64_t first_entry, const uint32_t* keys, const uint32_t* hist,
                                       uint32_t* scratch, int scratch_words, MergeSmem<NT>& sm) {
  const int32_t* pool = a.pool ? a.pool + (int64_t)b * a.pool_len + first_entry : nullptr;
  const bool tr = a.trace && b == 0 && chunk == 0 && threadIdx.x == 0;
  const int n_real = (int)sm.n_real;
  const int K = a.pool_out > 0 ? a.pool_out : a.topk;
  auto entry_of = [&](int i) { return pool ? pool[i] : (int32_t)(first_entry + i); };
  if (a.n_chunks == 1 && a.pool_out == 0) {
    // one chunk holds the whole sequence: its top-k is the answer
    int32_t* oi = a.out_idx + (int64_t)b * a.topk;
    const int kt = min(a.topk, n_real);
    SelSrc src{};
    src.key = keys;
    src.pool = pool;
    src.first = first_entry;
    select_ordered<NT>(src, n_elem, kt, 0u, 32, 0, oi, nullptr, sm.sel);
#pragma unroll 1
    for (int i = kt + threadIdx.x; i < a.topk; i += NT) oi[i] = -1;
    pdl_launch_dependents();
    return;
  }
  const long long t0 = clock64();
  uint32_t* seq = a.seq_state + (int64_t)b * kSeqWords;
  uint32_t* gh = a.ghist + (int64_t)b * kBins;
  // 1. publish the histogram of the real keys
  const int bmin = n_real > 0 ? (int)key_bin(sm.kmin) : 0;
  const int bmax = n_real > 0 ? (int)key_bin(sm.kmax) : -1;
#pragma unroll 1
  for (int v = bmin + (int)threadIdx.x; v <= bmax; v += NT) {
    const uint32_t c = hist[v];
    if (c) atomicAdd(gh + v, c);
  }
  if (threadIdx.x == 0 && n_real > 0) {
    atomicMax(seq + 1, (uint32_t)bmax + 1u);
    atomicMax(seq + 2, (uint32_t)(kBins - bmin));
  }
  trace_at(a.st, tr, 10, t0);
  // 2. lower bound on the sequence's threshold bin (no wait for this chunk's
  // own additions: the bound holds for any snapshot).  The scan starts at
  // this chunk's own top bin: keys of other chunks above it are left out,
  // which only lowers the counts and so keeps the bound valid.
  uint32_t bound = 0;
  if (n_real > K) bound = chunk_bound<NT>(gh, hist, bmax + 1, (uint32_t)K, sm);
  const uint32_t lo_key = bound << kBinShift;
  trace_at(a.st, tr, 11, t0);
  // 3. candidates (real keys >= lo_key) in entry order
  const int64_t slot0 = ((int64_t)b * a.n_chunks + chunk) * a.chunk;
  uint32_t* ck = a.cand_key + slot0;
  int32_t* ci = a.cand_idx + slot0;
  {
    // warp w takes a contiguous range of 32-key groups: count, one barrier
    // for the warps' offsets, then write in order
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = NT / 32;
    const int groups = (n_elem + 31) / 32, gper = (groups + kWarps - 1) / kWarps;
    const int i0 = min(n_elem, warp * gper * 32), i1 = min(n_elem, (warp + 1) * gper * 32);
    auto take = [&](int i) {
      const uint32_t u = i < i1 ? keys[i] : 0u;
      return u != 0u && u >= lo_key;
    };
    uint32_t cnt = 0;
#pragma unroll 1
    for (int i = i0 + lane; i - lane < i1; i += 128) {
      bool f[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) f[q] = take(i + 32 * q);
#pragma unroll
      for (int q = 0; q < 4; ++q) cnt += __popc(__ballot_sync(0xffffffffu, f[q]));
    }
    if (lane == 0) sm.wcnt[warp] = cnt;
    __syncthreads();
    uint32_t pos = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t c = sm.wcnt[w];
      pos += w < warp ? c : 0u;
      tot += c;
    }
#pragma unroll 1
    for (int i = i0 + lane; i - lane < i1; i += 128) {
      bool f[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) f[q] = take(i + 32 * q);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t bal = __ballot_sync(0xffffffffu, f[q]);
        if (f[q]) {
          const uint32_t at = pos + __popc(bal & ((1u << lane) - 1u));
          ck[at] = keys[i + 32 * q];
          ci[at] = entry_of(i + 32 * q);
        }
        pos += __popc(bal);
      }
    }
    if (threadIdx.x == 0)
      reinterpret_cast<uint2*>(a.ccount)[(int64_t)b * a.n_chunks + chunk] = make_uint2(tot, (uint32_t)n_real);
  }
  trace_at(a.st, tr, 12, t0);
  if (tr) {
    a.st->pad[29] = (int32_t)bound;
    a.st->pad[30] = (int32_t)reinterpret_cast<uint2*>(a.ccount)[(int64_t)b * a.n_chunks + chunk].x;
  }
  __threadfence();
  __syncthreads();
  pdl_launch_dependents();   // the next kernel may take the SMs this grid frees
  if (threadIdx.x == 0) sm.ticket = (int)atomicAdd(seq, 1u);
  __syncthreads();
  if (sm.ticket != a.n_chunks - 1) return;
  __threadfence();
  merge_and_emit<NT, BM>(a, b, sm, scratch, scratch_words, bound);
}

}  // namespace ckv

// csa_index_topk: Lightning-indexer scores and exact top-k per sequence.
//
// "DeepSeek-V4 KV Cache 深度分析", §四: the 128-d indexer query of the current
// token is scored against every compressed block's indexer key and the top-k
// blocks are kept; the indexer's QK activations are held and computed in FP4.
// Score (workload definition): s_j = sum_h w_h * ReLU(q_h . k_j) on the
// dequantised values; for FP4 keys the query is block-quantised first.
//
// Grid (chunk, sequence).  Each CTA scores one chunk of entries, histograms
// their keys, and writes the keys above a lower bound on the sequence's
// threshold (from the sequence histogram in the workspace) as its
// candidates; the last CTA of a sequence to finish (atomic ticket, no
// spinning) merges them into the exact top-K, and for a CSA2 Full layer also
// the top-k of that pool (topk_merge.cuh).  Candidate lists are in ascending
// entry order, so the merge's ordered compaction resolves ties towards the
// lower index.
//
// Scoring engines:
//   * score_simt: CUDA-core FMAs on dequantised values (BF16 keys, the CSA2
//     Reindex pass over a candidate pool, and FP4 keys when the block-scaled
//     tensor-core scorer is not used);
//   * the block-scaled tcgen05 scorer lives in indexer_umma.cu.

#include <cstddef>

#include "topk_merge.cuh"
#include "hadamard.cuh"

namespace ckv {

constexpr int kIdxThreads = 512;

struct IndexSmem {
  float q[kMaxHI * kIdxDim];       // dequantised indexer query
  float w[kMaxHI];
  uint32_t keys[kMaxChunk];        // scores of this chunk as order keys (0 = no entry)
  uint32_t hist[kBins];            // their histogram (top kBinBits bits)
  float part[kIdxThreads];         // half-head partial scores (two threads per key)
  MergeSmem<kIdxThreads> m;
};
static_assert(offsetof(IndexSmem, hist) == offsetof(IndexSmem, keys) + kMaxChunk * 4,
              "keys and hist are one block of merge scratch");

// Dequantised indexer query into shared memory: FP4 keys -> the query is
// quantised with the E2M1 + E4M3/16 block quantiser (the same arithmetic as
// the append path) and its exact values stored; BF16 keys -> the BF16 values.
__device__ void load_query(const IndexArgs& a, int b, float* q, float* w) {
  if (a.fmt == CKV_FMT_FP4H) {
    // Hadamard-rotated keys: each warp rotates and quantises whole heads
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int h = threadIdx.x >> 5; h < a.HI; h += kIdxThreads / 32) {
      const uint2 raw = *reinterpret_cast<const uint2*>(a.q_idx + ((int64_t)b * a.HI + h) * kIdxDim + lane * 4);
      float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                    __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
      hadamard128_warp(v, lane);
      uint8_t sc;
      const uint32_t c = fp4_quant_lane4(v, sc);
      const float s = e4m3_value(sc);
#pragma unroll
      for (int i = 0; i < 4; ++i) q[h * kIdxDim + lane * 4 + i] = e2m1_value((c >> (4 * i)) & 0xFu) * s;
    }
    for (int t = threadIdx.x; t < a.HI; t += kIdxThreads) w[t] = a.w[(int64_t)b * a.HI + t];
    return;
  }
  for (int t = threadIdx.x; t < a.HI * 8; t += kIdxThreads) {
    const int h = t >> 3, blk = t & 7;
    const __nv_bfloat16* src = a.q_idx + ((int64_t)b * a.HI + h) * kIdxDim + blk * 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    const uint4 x0 = s4[0], x1 = s4[1];
    const uint32_t wd[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(wd[i] << 16);
      v[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
    }
    if (a.fmt == CKV_FMT_FP4) {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const float s = e4m3_value(e4m3_code(__fdiv_rn(amax, 6.0f)));
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = s > 0.f ? e2m1_value(e2m1_code(__fdiv_rn(v[i], s))) * s : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) q[h * kIdxDim + blk * 16 + i] = v[i];
  }
  for (int t = threadIdx.x; t < a.HI; t += kIdxThreads) w[t] = a.w[(int64_t)b * a.HI + t];
}

// Score of one key, block by block (16 channels); block blk + 1's bytes are
// loaded while block blk is multiplied, so one memory round trip per key is
// exposed rather than one per block.
template <int HMAX>
__device__ __forceinline__ float score_simt(const IndexArgs& a, int b, int64_t entry,
                                            const float* q, const float* w, int h0 = 0) {
  // heads h0 .. h0 + HMAX - 1 (those below HI)
  float acc[HMAX];
#pragma unroll
  for (int h = 0; h < HMAX; ++h) acc[h] = 0.f;
  int64_t row = plane_row(a.bt, a.page, a.bt_cols, a.cap, b, entry);
  if (row < 0 || row >= a.rows) {   // a page id beyond the plane: scored as row 0, recorded
    report(a.st, CKV_ERR_DEVICE_BOUNDS, (int)entry);
    row = 0;
  }
  const bool fp4 = a.fmt == CKV_FMT_FP4 || a.fmt == CKV_FMT_FP4H;
  auto fetch = [&](int blk, uint4& x0, uint4& x1, uint32_t& sc) {
    if (fp4) {
      const uint2 d = *reinterpret_cast<const uint2*>(a.kdata + row * 64 + blk * 8);
      x0 = make_uint4(d.x, d.y, 0u, 0u);
      x1 = make_uint4(0u, 0u, 0u, 0u);
      sc = a.kscale[row * 8 + blk];
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(a.kdata + row * 256 + blk * 32);
      x0 = p[0];
      x1 = p[1];
      sc = 0u;
    }
  };
  uint4 n0, n1;
  uint32_t ns;
  fetch(0, n0, n1, ns);
#pragma unroll 1
  for (int blk = 0; blk < 8; ++blk) {
    const uint4 x0 = n0, x1 = n1;
    const uint32_t xs = ns;
    if (blk + 1 < 8) fetch(blk + 1, n0, n1, ns);
    float kv[16];
    if (fp4) {
      // hardware E2M1 decode, two codes (low nibble first) per byte; the
      // f16 values are exact, the f32 products too
      const float s = e4m3_value((uint8_t)xs);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 lo = __half22float2(__half2(__nv_cvt_fp4x2_to_halfraw2(
            (__nv_fp4x2_storage_t)((x0.x >> (8 * i)) & 0xFF), __NV_E2M1)));
        const float2 hi = __half22float2(__half2(__nv_cvt_fp4x2_to_halfraw2(
            (__nv_fp4x2_storage_t)((x0.y >> (8 * i)) & 0xFF), __NV_E2M1)));
        kv[2 * i] = lo.x * s;
        kv[2 * i + 1] = lo.y * s;
        kv[8 + 2 * i] = hi.x * s;
        kv[8 + 2 * i + 1] = hi.y * s;
      }
    } else {
      const uint32_t wd[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        kv[2 * i] = __uint_as_float(wd[i] << 16);
        kv[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int h = 0; h < HMAX; ++h) {
      if (h0 + h < a.HI) {
        const float4* qq = reinterpret_cast<const float4*>(q + (h0 + h) * kIdxDim + blk * 16);
        float r = acc[h];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 v = qq[j];
          r = fmaf(v.x, kv[4 * j], r);
          r = fmaf(v.y, kv[4 * j + 1], r);
          r = fmaf(v.z, kv[4 * j + 2], r);
          r = fmaf(v.w, kv[4 * j + 3], r);
        }
        acc[h] = r;
      }
    }
  }
  float s = 0.f;
#pragma unroll
  for (int h = 0; h < HMAX; ++h)
    if (h0 + h < a.HI) s = fmaf(w[h0 + h], fmaxf(acc[h], 0.f), s);
  return s;
}

// HMAX: the head count rounded up to 8, 16, 32 or 64; the head loops are
// unrolled to HMAX, so a few heads do not pay for sixty-four.
template <int HMAX>
__global__ void __launch_bounds__(kIdxThreads, 1) index_topk_simt_kernel(IndexArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  IndexSmem& sm = *reinterpret_cast<IndexSmem*>(smem_raw);
  pdl_wait();
  const int b = blockIdx.y, chunk = blockIdx.x;
  const bool tr = a.trace && b == 0 && chunk == 0 && threadIdx.x == 0;
  const long long t0 = clock64();
  const int ncomp = min(a.n_comp[b], a.n_comp_max);
  load_query(a, b, sm.q, sm.w);
  merge_smem_init<kIdxThreads>(sm.m);
  for (int i = threadIdx.x; i < kBins / 4; i += kIdxThreads)
    reinterpret_cast<uint4*>(sm.hist)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  trace_at(a.st, tr, 0, t0);

  int n_elem;
  int64_t first = 0;
  const int32_t* pool = nullptr;
  if (a.pool) {
    // Reindex: chunk `chunk` of the candidate list; entries come from it
    first = (int64_t)chunk * a.chunk;
    pool = a.pool + (int64_t)b * a.pool_len + first;
    n_elem = (int)max((int64_t)0, min((int64_t)a.chunk, (int64_t)a.pool_len - first));
  } else {
    first = (int64_t)chunk * a.chunk;
    n_elem = (int)max((int64_t)0, min((int64_t)a.chunk, (int64_t)ncomp - first));
  }
  uint32_t mine = 0;
  bool split = false;
  if constexpr (HMAX == 64) {
    split = n_elem <= kIdxThreads / 2 && a.HI > 32;
    if (split) {
      // few keys (a Reindex chunk): two threads per key, 32 heads each
      const int k = threadIdx.x & (kIdxThreads / 2 - 1), hh = threadIdx.x / (kIdxThreads / 2);
      float part = 0.f;
      int64_t e = -1;
      if (k < n_elem) {
        e = pool ? (int64_t)pool[k] : first + k;
        if (e >= 0 && e < ncomp) part = score_simt<32>(a, b, e, sm.q, sm.w, 32 * hh);
      }
      sm.part[threadIdx.x] = part;
      __syncthreads();
      if (hh == 0 && k < n_elem) {
        uint32_t key = 0u;
        if (e >= 0 && e < ncomp) {
          const float sc = sm.part[k] + sm.part[k + kIdxThreads / 2];
          key = score_key(sc);
          if (a.dbg) a.dbg[(int64_t)b * a.n_comp_max + e] = sc;
          ++mine;
        } else if (e >= ncomp && pool) {
          report(a.st, CKV_ERR_DEVICE_BOUNDS, (int)e);
        }
        sm.keys[k] = key;
      }
    }
  }
  for (int i = threadIdx.x; !split && i < n_elem; i += kIdxThreads) {
    int64_t e = pool ? (int64_t)pool[i] : first + i;
    uint32_t key = 0u;
    if (e >= 0 && e < ncomp) {
      const float s = score_simt<HMAX>(a, b, e, sm.q, sm.w);
      key = score_key(s);
      if (a.dbg) a.dbg[(int64_t)b * a.n_comp_max + e] = s;
      ++mine;
    } else if (e >= ncomp && pool) {
      report(a.st, CKV_ERR_DEVICE_BOUNDS, (int)e);
    }
    sm.keys[i] = key;
  }
  atomicAdd(&sm.m.n_real, mine);
  __syncthreads();
  // histogram and range of the real keys
  {
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    for (int i = threadIdx.x; i < n_elem; i += kIdxThreads) {
      const uint32_t u = sm.keys[i];
      if (u != 0u) {
        atomicAdd(&sm.hist[key_bin(u)], 1u);
        kmin = min(kmin, u);
        kmax = max(kmax, u);
      }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if ((threadIdx.x & 31) == 0) {
      atomicMin(&sm.m.kmin, kmin);
      atomicMax(&sm.m.kmax, kmax);
    }
  }
  __syncthreads();
  trace_at(a.st, tr, 9, t0);
  chunk_select_and_merge<kIdxThreads>(a, b, chunk, n_elem, first, sm.keys, sm.hist, sm.keys,
                                      kMaxChunk + kBins, sm.m);
}

size_t index_smem_bytes() { return sizeof(IndexSmem); }

cudaError_t launch_index_simt(const IndexArgs& a, cudaStream_t stream) {
  using KernelFn = void (*)(IndexArgs);
  const KernelFn ks[4] = {index_topk_simt_kernel<8>, index_topk_simt_kernel<16>,
                          index_topk_simt_kernel<32>, index_topk_simt_kernel<64>};
  static DeviceOnce once;
  const cudaError_t e = once_per_device(once, [&](int) {
    for (KernelFn k : ks) {
      const cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)sizeof(IndexSmem));
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  static_assert(kMaxHI <= 64, "the widest instance covers every head count");
  const KernelFn kern = a.HI <= 8 ? ks[0] : a.HI <= 16 ? ks[1] : a.HI <= 32 ? ks[2] : ks[3];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.B);
  cfg.blockDim = dim3(kIdxThreads);
  cfg.dynamicSmemBytes = sizeof(IndexSmem);
  cfg.stream = stream;
  cudaLaunchAttribute at[1] = {pdl_attribute()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace ckv

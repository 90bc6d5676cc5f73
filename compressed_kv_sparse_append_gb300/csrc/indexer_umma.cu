// Block-scaled tcgen05 scorer of csa_index_topk for FP4 indexer keys.
//
// "DeepSeek-V4 KV Cache 深度分析", §四 (and the paper's Section 5.2.1 quoted
// there): the indexer's QK activations are cached, loaded and computed in FP4.
// Keys and query are E2M1 with one E4M3 scale per 16 channels ("V4.1-Flash
// 공개", 핵심 내용: the same block format as the FP4 main KV), which is exactly
// the operand format of tcgen05.mma kind::mxf4nvf4 with scale_vec::4X: the
// tensor core applies both scales per 16-element block and accumulates in
// f32, so the FP4 bytes go from HBM to the tensor core untouched.
//
// Per CTA: one chunk of C keys of one sequence (for a CSA2 Reindex pass: C
// entries of the sequence's candidate pool).
//   warp 0   producer: 128-key tiles of packed codes (SWIZZLE_64B) and
//            their scale bytes into a kUStages-deep shared-memory ring,
//            starting as soon as the previous kernel is done (the other
//            warps quantise the query meanwhile) -- streamed by TMA, or,
//            for a pool, gathered row by row with cp.async;
//   warps 1 and 14 MMA issuers, of the even and the odd tiles (warp 1 owns
//            TMEM): D[128 keys x 64 heads] (f32, four buffers, so the MMA
//            runs up to three tiles ahead of the epilogue) = keys (A,
//            M = 128) x query (B, N = 64), K = 128 in two block-scaled steps.
//            A single issuing thread is a serial chain of waits, descriptor
//            arithmetic and MMA issues (each tcgen05.mma or commit costs it
//            tens of cycles); two of them, on different SM sub-partitions
//            and with disjoint stages, accumulators and barriers, keep the
//            tensor core fed twice as fast;
//   warps 6-9 move each tile's key scales into TMEM (lane = key), running
//            ahead of the MMA by up to the ring depth;
//   warps 2-5 epilogue: read D back (one key per thread), form
//            s = sum_h w_h ReLU(d_h) in f32, and count its key in the
//            chunk's shared-memory histogram.
// The scores stay in shared memory; the candidate bound and the cross-chunk
// merge are those of topk_merge.cuh.

#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "tmap.cuh"
#include "topk_merge.cuh"
#include "hadamard.cuh"

namespace ckv {

namespace {

// warp 0 TMA, warps 1 and 14 MMA (even / odd tiles), warps 2-5 and 10-13
// epilogue (even / odd tiles), warps 6-9 scale movers
constexpr int kUThreads = 480;
constexpr int kUStages = 14;
constexpr int kUTile = 128;
constexpr uint32_t kDataBytes = kUTile * 64;                 // 8 KB
constexpr uint32_t kScaleBytes = kUTile * 8;                 // 1 KB
// The ring, the chunk's keys and their histogram come first and are
// contiguous: once the chunk's candidates are written they are dead and
// serve the merge as one scratch block.
constexpr uint32_t kOffData = 0;
constexpr uint32_t kOffScale = kOffData + kUStages * kDataBytes;
constexpr uint32_t kOffKeys = kOffScale + kUStages * kScaleBytes;  // u32 [kMaxChunk]
constexpr uint32_t kOffHist = kOffKeys + kMaxChunk * 4;            // u32 [kBins]
constexpr uint32_t kOffQ = (kOffHist + kBins * 4 + 1023) & ~1023u; // 64 rows x 64 B
constexpr uint32_t kOffQs = kOffQ + 64 * 64;                       // 64 x 8 scale bytes
constexpr uint32_t kOffW = kOffQs + 64 * 8;                        // 64 f32
constexpr uint32_t kOffMerge = kOffW + 64 * 4;
constexpr uint32_t kOffBar = (kOffMerge + sizeof(MergeSmem<kUThreads>) + 7) & ~7u;
constexpr int kLongSequenceEntries = 131072;   // above: the kernel instance with the bitmap output
constexpr int kDBuf = 4;          // TMEM accumulators: the MMA runs up to 3 tiles ahead
constexpr int kNumBarU = 3 * kUStages + 2 * kDBuf;
constexpr uint32_t kOffSlotU = kOffBar + kNumBarU * 8;
constexpr uint32_t kSmemU = kOffSlotU + 16 + 1024;
static_assert(kOffQ % 1024 == 0, "operand tiles 1024-aligned");
static_assert(kUStages % 2 == 0 && kDBuf % 2 == 0, "each MMA issuer owns alternate stages and accumulators");
static_assert(kSmemU <= 232448, "fits in shared memory");
// The merge's shared-memory scratch: ring, keys and histogram (dead by then).
constexpr int kMergeScratchWords = (int)((kOffHist + kBins * 4) / 4);

constexpr uint32_t kTmemU = 512;
constexpr uint32_t kColD = 0;          // kDBuf 64-column accumulators
constexpr uint32_t kColSFA = 64 * kDBuf;   // 8 columns per stage
constexpr uint32_t kColSFB = kColSFA + 8 * kUStages;   // 8 columns
static_assert(kColSFB + 8 <= kTmemU, "scale columns of every stage and the query's fit");
constexpr uint32_t kIdescNvf4 = idesc_nvf4(128, 64);

enum { BU_FULL = 0, BU_EMPTY = kUStages, BU_SFA = 2 * kUStages, BU_DFULL = 3 * kUStages,
       BU_DEMPTY = 3 * kUStages + kDBuf };

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// cp.async of `bytes` (8 or 16) from global to shared; src_bytes = 0 reads
// nothing and writes zeros.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async8_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// Arrive on `bar` once every cp.async this thread issued before has landed
// (the arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 16-byte chunk c (0..3) of row r of a 64-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

}  // namespace

struct UmmaIndexArgs {
  IndexArgs a;
  int64_t row_limit;  // B * cap (rows of the key plane)
};

template <bool BM>
__global__ void __launch_bounds__(kUThreads, 1)
    index_topk_umma_kernel(const __grid_constant__ CUtensorMap map_data,
                           const __grid_constant__ CUtensorMap map_scale, UmmaIndexArgs ua) {
  const IndexArgs& a = ua.a;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* g = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(g + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(g + kOffSlotU);
  uint32_t* keys = reinterpret_cast<uint32_t*>(g + kOffKeys);
  uint32_t* hist = reinterpret_cast<uint32_t*>(g + kOffHist);
  float* wsm = reinterpret_cast<float*>(g + kOffW);
  MergeSmem<kUThreads>& msm = *reinterpret_cast<MergeSmem<kUThreads>*>(g + kOffMerge);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // barriers and TMEM first: they touch only this CTA's own resources; global
  // memory (inputs included) only after the previous kernel is done
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kUStages; ++s) {
      // a gathered tile completes with the 32 producer lanes' cp.async
      // arrivals, a streamed one with one transaction-counted TMA arrival
      mbar_init(&bars[BU_FULL + s], a.pool ? 32 : 1);
      mbar_init(&bars[BU_EMPTY + s], 1);
      mbar_init(&bars[BU_SFA + s], 128);
    }
    for (int d = 0; d < kDBuf; ++d) {
      mbar_init(&bars[BU_DFULL + d], 1);
      mbar_init(&bars[BU_DEMPTY + d], 128);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, kTmemU);
  merge_smem_init<kUThreads>(msm);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  pdl_wait();
  const int b = blockIdx.y, chunk = blockIdx.x;
  const int ncomp = min(a.n_comp[b], a.n_comp_max);
  const int64_t c0 = (int64_t)chunk * a.chunk;
  // Reindex (a.pool): chunk `chunk` of the sequence's candidate list, whose
  // entries name the keys; otherwise keys c0 .. of the plane
  const int32_t* pl = a.pool ? a.pool + (int64_t)b * a.pool_len + c0 : nullptr;
  const int64_t n_avail = a.pool ? (int64_t)a.pool_len - c0 : (int64_t)ncomp - c0;
  const int n_elem = (int)max((int64_t)0, min((int64_t)a.chunk, n_avail));
  const int T = (n_elem + kUTile - 1) / kUTile;
  const int64_t row0 = (int64_t)b * a.cap + c0;
  volatile int* abort_p = &abort_flag;
  const bool tr = a.trace && b == 0 && chunk == 0;
  const long long tr0 = clock64();

  if (warp == 0 && pl) {
    // ----------------------------------------------- gathered key rows ----
    // Lane l gathers keys l, l + 32, l + 64, l + 96 of each tile: the 64
    // code bytes (four 16-byte copies to their SW64 places) and the 8 scale
    // bytes of the key's row; an empty or out-of-range entry copies zeros.
    // The stage completes with every lane's cp.async arrival.
    const uint8_t* kd = static_cast<const uint8_t*>(a.kdata);
    const uint8_t* ks = static_cast<const uint8_t*>(a.kscale);
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
      const int s = t % kUStages;
      bool ok = true;
      if (lane == 0 && t >= kUStages)
        ok = mbar_wait_cta(&bars[BU_EMPTY + s], ((t / kUStages) + 1) & 1, a.st, abort_p, 11);
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
      int32_t e[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = t * kUTile + lane + 32 * k;
        e[k] = i < n_elem ? __ldg(pl + i) : -1;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = lane + 32 * k;
        int64_t row = -1;
        if (e[k] >= ncomp) report(a.st, CKV_ERR_DEVICE_BOUNDS, e[k]);
        else if (e[k] >= 0) row = plane_row(a.bt, a.page, a.bt_cols, a.cap, b, e[k]);
        if (row >= ua.row_limit) {   // a page id beyond the plane
          report(a.st, CKV_ERR_DEVICE_BOUNDS, e[k]);
          row = -1;
        }
        const uint32_t nb = row >= 0 ? 16u : 0u;
        const int64_t rr = row >= 0 ? row : 0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          cp_async16_zfill(base + kOffData + s * kDataBytes + sw64(r, c), kd + rr * 64 + c * 16, nb);
        cp_async8_zfill(base + kOffScale + s * kScaleBytes + r * 8, ks + rr * 8, nb >> 1);
      }
      cp_async_arrive_noinc(&bars[BU_FULL + s]);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");   // nothing in flight past this point
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA ----
    // The key stream does not depend on the query: it starts at once, while
    // the other warps prepare the query.
    // A paged plane: the whole warp fetches the pages of the next 32 tiles
    // (a 128-key tile lies in one page), lane 0 issues.
    int pg_reg = 0;
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
      const int s = t % kUStages;
      bool ok = true;
      if (lane == 0 && t >= kUStages)
        ok = mbar_wait_cta(&bars[BU_EMPTY + s], ((t / kUStages) + 1) & 1, a.st, abort_p, 11);
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
      int64_t row = row0 + (int64_t)t * kUTile;
      if (a.bt) {
        if ((t & 31) == 0) {
          const int64_t p0 = c0 + (int64_t)(t + lane) * kUTile;
          pg_reg = t + lane < T ? __ldg(a.bt + (int64_t)b * a.bt_cols + (int)(p0 / a.page)) : 0;
        }
        const int pg = __shfl_sync(0xffffffffu, pg_reg, t & 31);
        const int64_t pos = c0 + (int64_t)t * kUTile;
        row = (int64_t)pg * a.page + pos % a.page;
      }
      if (lane == 0) {
        mbar_expect_tx(&bars[BU_FULL + s], kDataBytes + kScaleBytes);
        tma_load_2d(base + kOffData + s * kDataBytes, &map_data, 0, (int)row, &bars[BU_FULL + s]);
        tma_load_2d(base + kOffScale + s * kScaleBytes, &map_scale, 0, (int)(row >> 1),
                    &bars[BU_FULL + s]);
      }
    }
    __syncwarp();
  } else {
    // ---- warps 1-13: FP4 query (B operand) + its scales, head weights, an
    // empty histogram
    const int t9 = tid - 32;
    if (a.fmt == CKV_FMT_FP4H) {
      // Hadamard-rotated keys: each warp rotates and quantises whole heads
      // (4 channels per lane); lane l's two code bytes are bytes 2l, 2l + 1
      // of row h of the SW64 tile, its block l / 4's scale goes to the scale
      // table
#pragma unroll 1
      for (int h = warp - 1; h < 64; h += kUThreads / 32 - 1) {
        uint32_t c = 0;
        uint8_t sc = 0;
        if (h < a.HI) {
          const uint2 raw = *reinterpret_cast<const uint2*>(a.q_idx + ((int64_t)b * a.HI + h) * kIdxDim + lane * 4);
          float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                        __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
          hadamard128_warp(v, lane);
          c = fp4_quant_lane4(v, sc);
        }
        *reinterpret_cast<uint16_t*>(g + kOffQ + sw64(h, lane >> 3) + ((2 * lane) & 15)) = (uint16_t)c;
        if ((lane & 3) == 0) g[kOffQs + h * 8 + (lane >> 2)] = sc;
      }
    }

    constexpr int kQItems = (64 * 8 + kUThreads - 33) / (kUThreads - 32);   // 16-channel blocks per thread
    const bool plain_q = a.fmt != CKV_FMT_FP4H;
    uint4 qraw[kQItems][2];
#pragma unroll
    for (int k = 0; k < kQItems; ++k) {
      const int j = t9 + k * (kUThreads - 32), h = j >> 3, blk = j & 7;
      qraw[k][0] = qraw[k][1] = make_uint4(0u, 0u, 0u, 0u);
      if (plain_q && j < 64 * 8 && h < a.HI) {
        const uint4* s4 = reinterpret_cast<const uint4*>(a.q_idx + ((int64_t)b * a.HI + h) * kIdxDim + blk * 16);
        qraw[k][0] = s4[0];
        qraw[k][1] = s4[1];
      }
    }
    const float wv = (t9 < 64 && t9 < a.HI) ? a.w[(int64_t)b * a.HI + t9] : 0.f;
#pragma unroll
    for (int k = 0; k < kQItems; ++k) {
      const int j = t9 + k * (kUThreads - 32), h = j >> 3, blk = j & 7;
      if (j >= 64 * 8 || !plain_q) break;
      uint32_t lo = 0, hi = 0;
      uint8_t sc = 0;
      if (h < a.HI) {
        const uint4 x0 = qraw[k][0], x1 = qraw[k][1];
        const uint32_t wd[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float v[16];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = __uint_as_float(wd[i] << 16);
          v[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        sc = e4m3_code(__fdiv_rn(amax, 6.0f));
        const float s = e4m3_value(sc);
        if (s > 0.f) {
#pragma unroll
          for (int i = 0; i < 8; ++i) lo |= e2m1_code(__fdiv_rn(v[i], s)) << (4 * i);
#pragma unroll
          for (int i = 0; i < 8; ++i) hi |= e2m1_code(__fdiv_rn(v[8 + i], s)) << (4 * i);
        } else {
          sc = 0;
        }
      }
      // row h, bytes [8 blk, 8 blk + 8) of the SW64 tile
      *reinterpret_cast<uint2*>(g + kOffQ + sw64(h, blk >> 1) + (blk & 1) * 8) = make_uint2(lo, hi);
      g[kOffQs + h * 8 + blk] = sc;
    }
    if (t9 < 64) wsm[t9] = wv;
    for (int i = t9; i < kBins / 4; i += kUThreads - 32)
      reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    asm volatile("bar.sync 1, %0;" ::"r"(kUThreads - 32) : "memory");
    if (warp >= 2 && warp < 6) {
      // query scales -> TMEM (B operand scales): lane 32q + r, column j holds
      // the four block scales (one 32-bit word per K step) of query row 32j + r.
      const int qd = warp & 3;
      const int m = qd * 32 + lane;
      const uint32_t lb = (uint32_t)(qd * 32) << 16;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = 32 * j + (m & 31);
          v[j] = row < 64 ? *reinterpret_cast<const uint32_t*>(g + kOffQs + row * 8 + ks * 4) : 0u;
        }
        tmem_st4(tmem + lb + kColSFB + 4 * ks, v[0], v[1], v[2], v[3]);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"r"(kUThreads - 32) : "memory");
    tc_fence_after();
    if (tid == 32) trace_at(a.st, tr, 0, tr0);

    if (warp == 1 || warp == 14) {
      // ------------------------------------------------------------ MMA ----
      // Issuer `par` takes tiles par, par + 2, ...: their stages (kUStages is
      // even), accumulators and barriers are its own.
      if (lane == 0) {
        const int par = warp == 1 ? 0 : 1;
        // descriptors: the stage and K step only move the start address,
        // whose field (address >> 4, 14 bits) never carries
        const uint64_t da0 = smem_desc(base + kOffData, 16, 512, 4);
        const uint64_t db0 = smem_desc(base + kOffQ, 16, 512, 4);
        const uint64_t db1 = smem_desc(base + kOffQ + 32, 16, 512, 4);
#pragma unroll 1
        for (int t = par; t < T; t += 2) {
          const int s = t % kUStages, d = t % kDBuf;
          if (!mbar_wait_cta(&bars[BU_SFA + s], (t / kUStages) & 1, a.st, abort_p, 12)) break;
          if (t >= kDBuf && !mbar_wait_cta(&bars[BU_DEMPTY + d], ((t / kDBuf) + 1) & 1, a.st, abort_p, 13))
            break;
          tc_fence_after();
          // gathered tiles were written by cp.async (the generic proxy); the
          // MMA reads them through the async proxy
          if (pl) fence_proxy_async_smem();
          if (t < 8) trace_at(a.st, tr, 32 + t, tr0);
          const uint64_t da = da0 + ((s * kDataBytes) >> 4);
          const uint32_t dt = tmem + kColD + 64 * d, sfa = tmem + kColSFA + 8 * s;
          umma_nvf4(dt, da, db0, kIdescNvf4, sfa, tmem + kColSFB, 0u);
          umma_nvf4(dt, da + 2, db1, kIdescNvf4, sfa + 4, tmem + kColSFB + 4, 1u);
          umma_commit(&bars[BU_DFULL + d]);
          umma_commit(&bars[BU_EMPTY + s]);
          if (t < 8) trace_at(a.st, tr, (par ? 56 : 13) + t / 2, tr0);
        }
      }
      __syncwarp();
    } else if (warp >= 6 && warp < 10) {
      // --------------------------------------------------- scale movers ----
      const int qd = warp & 3;
      const int m = qd * 32 + lane;
      const uint32_t lb = (uint32_t)(qd * 32) << 16;
      for (int t = 0; t < T; ++t) {
        const int s = t % kUStages;
        if (!mbar_wait_cta(&bars[BU_FULL + s], (t / kUStages) & 1, a.st, abort_p, 14)) break;
        const uint2 sc = *reinterpret_cast<const uint2*>(g + kOffScale + s * kScaleBytes + m * 8);
        tmem_st4(tmem + lb + kColSFA + 8 * s, sc.x, sc.x, sc.x, sc.x);
        tmem_st4(tmem + lb + kColSFA + 8 * s + 4, sc.y, sc.y, sc.y, sc.y);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[BU_SFA + s]);
        if (m == 0 && t < 8) trace_at(a.st, tr, 40 + t, tr0);
      }
    } else {
      // ------------------------------------------------------- epilogue ----
      // group 0 (warps 2-5) takes the even tiles (accumulator 0), group 1
      // (warps 10-13) the odd ones (accumulator 1): two warps per SM
      // sub-partition, so one's TMEM loads and FMAs overlap the other's
      const int qd = warp & 3;
      const int grp = warp >= 10 ? 1 : 0;
      const int m = qd * 32 + lane;                 // key of the tile = TMEM lane
      const uint32_t lb = (uint32_t)(qd * 32) << 16;
      uint32_t kmin = 0xFFFFFFFFu, kmax = 0u, n_mine = 0u;
      for (int t = grp; t < T; t += 2) {
        const int d = t % kDBuf;
        // the key's entry (its candidate-list value for a Reindex), read
        // before the wait so that its latency hides behind it
        const int i = t * kUTile + m;
        const int64_t ent = pl ? (i < n_elem ? (int64_t)__ldg(pl + i) : -1) : c0 + i;
        if (!mbar_wait_cta(&bars[BU_DFULL + d], (t / kDBuf) & 1, a.st, abort_p, 15)) break;
        tc_fence_after();
        if (m == 0 && t < 8) trace_at(a.st, tr, 48 + t, tr0);
        uint32_t r[64];
        tmem_ld32(tmem + lb + kColD + 64 * d, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(tmem + lb + kColD + 64 * d + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars[BU_DEMPTY + d]);
        // eight independent partial sums (one f32 FMA chain of 64 would
        // leave the single epilogue warp of each SM sub-partition waiting
        // on FMA latency), added in a fixed order
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h4 = 0; h4 < 16; ++h4) {
          const float4 wv = reinterpret_cast<const float4*>(wsm)[h4];
          const int j = (h4 & 1) * 4;
          acc[j] = fmaf(wv.x, fmaxf(__uint_as_float(r[4 * h4]), 0.f), acc[j]);
          acc[j + 1] = fmaf(wv.y, fmaxf(__uint_as_float(r[4 * h4 + 1]), 0.f), acc[j + 1]);
          acc[j + 2] = fmaf(wv.z, fmaxf(__uint_as_float(r[4 * h4 + 2]), 0.f), acc[j + 2]);
          acc[j + 3] = fmaf(wv.w, fmaxf(__uint_as_float(r[4 * h4 + 3]), 0.f), acc[j + 3]);
        }
        const float sc = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        if (m == 0 && t < 8) trace_at(a.st, tr, 1 + t, tr0);
        if (i < n_elem) {
          uint32_t key = 0u;   // an empty or out-of-range entry: no key
          if (ent >= 0 && ent < ncomp) {
            key = score_key(sc);
            atomicAdd(&hist[key_bin(key)], 1u);
            kmin = min(kmin, key);
            kmax = max(kmax, key);
            ++n_mine;
            if (a.dbg) a.dbg[(int64_t)b * a.n_comp_max + ent] = sc;
          }
          keys[i] = key;
        }
      }
      kmin = __reduce_min_sync(0xffffffffu, kmin);
      kmax = __reduce_max_sync(0xffffffffu, kmax);
      n_mine = __reduce_add_sync(0xffffffffu, n_mine);
      if (lane == 0) {
        atomicMin(&msm.kmin, kmin);
        atomicMax(&msm.kmax, kmax);
        atomicAdd(&msm.n_real, n_mine);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemU);
  }
  if (tid == 0) trace_at(a.st, tr, 9, tr0);
  if (tr && tid == 0) a.st->pad[24] = T;
  __syncthreads();
  // The merge's survivors use the pipeline ring, dead by then.
  chunk_select_and_merge<kUThreads, BM>(a, b, chunk, n_elem, c0, keys, hist,
                                        reinterpret_cast<uint32_t*>(g), kMergeScratchWords, msm);
}

bool index_umma_supported(const IndexArgs& a, int64_t batch_rows) {
  // FP4 keys, 64 heads max, the 2-D maps' row counts fit in int32; streamed
  // tiles (no pool) also need their scale rows to pair up (even cap) and a
  // page to hold whole tiles.  A Reindex pool gathers its rows one by one.
  const bool layout_ok = a.pool != nullptr || (a.bt ? a.page % kUTile == 0 : (a.cap % 2) == 0);
  return (a.fmt == CKV_FMT_FP4 || a.fmt == CKV_FMT_FP4H) && a.HI <= 64 && layout_ok &&
         batch_rows < (int64_t)1 << 31 && a.chunk % kUTile == 0 && tmap_encode_fn() != nullptr;
}

cudaError_t launch_index_umma(const IndexArgs& a, int64_t batch_rows, cudaStream_t stream) {
  static DeviceOnce once;
  const cudaError_t e = once_per_device(once, [](int) {
    cudaError_t r = cudaFuncSetAttribute(index_topk_umma_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemU);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(index_topk_umma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemU);
    return r;
  });
  if (e != cudaSuccess) return e;
  CUtensorMap md, ms;
  memset(&md, 0, sizeof(md));
  memset(&ms, 0, sizeof(ms));
  // streamed tiles only: a Reindex pool gathers its rows without the maps
  if (a.pool == nullptr &&
      (!encode_tmap_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.kdata, 64, (uint64_t)batch_rows, 64, 64,
                       (uint32_t)kUTile, CU_TENSOR_MAP_SWIZZLE_64B) ||
       !encode_tmap_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.kscale, 16, (uint64_t)(batch_rows / 2), 16,
                       16, (uint32_t)(kUTile / 2), CU_TENSOR_MAP_SWIZZLE_NONE)))
    return cudaErrorInvalidValue;
  UmmaIndexArgs ua;
  ua.a = a;
  ua.row_limit = batch_rows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.B);
  cfg.blockDim = dim3(kUThreads);
  cfg.dynamicSmemBytes = kSmemU;
  cfg.stream = stream;
  cudaLaunchAttribute at[1] = {pdl_attribute()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // Long sequences stage more candidates than one ordered pass of the merge
  // takes at once: their instance writes the output from bitmaps.
  const bool long_seq = a.n_comp_max > kLongSequenceEntries;
  return cudaLaunchKernelEx(&cfg, long_seq ? index_topk_umma_kernel<true> : index_topk_umma_kernel<false>,
                            md, ms, ua);
}

}  // namespace ckv

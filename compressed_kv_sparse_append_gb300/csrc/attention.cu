// csa_sparse_attn / hca_attn: shared-KV decode attention on tcgen05.
//
// "DeepSeek-V4 KV Cache 深度分析": §五 -- each compressed entry is both key
// and value (o = sum_j a_j C_j); §十一 -- Attention(Q, selected) followed by
// the 128-token window; §三 -- HCA attends densely to every ratio-128 entry
// plus the window.  One softmax over the union of the rows (no sink).
//
// Decomposition (per sequence b, one thread-block cluster of 2G CTAs):
//   * CTA (pair p, half c) owns latent dims [256c, 256c + 256).  TMEM:
//     O_c = 128 heads x 256 f32 (columns 0..255), Q_c as the bf16 A operand
//     (columns 256..383), two 128 x 64 f32 score buffers S (384..511); the
//     softmax writes P (bf16) over the first half of its S buffer and the
//     P.E product reads it from there, so neither Q nor P costs shared-memory
//     bandwidth.
//   * Pair p walks a contiguous range of 64-row tiles (selected entries, then
//     window slots).  For each tile both CTAs compute S_c = Q_c . E_c^T
//     (K = 256), swap S_c through distributed shared memory and add, so both
//     hold the same S bit for bit and run the same online softmax; then each
//     accumulates O_c += P . E_c (N = 256).
//   * The G pairs merge (m, l, O) in the cluster at the end: CTA (p, c)
//     finalises latent columns [256c + p*256/G, ...) from the G partial
//     accumulators of half c read over DSMEM.
// Warp roles: warp 0 issues TMA for contiguous BF16 tiles (HCA); warps 1-4
// gather + dequantise rows of the other formats (or zero the rows past the
// end of a partial TMA tile); warp 5 owns TMEM and issues every tcgen05.mma;
// warps 6-9 run the softmax, one head row per thread (warp % 4 = TMEM lane
// quarter).  Every wait is a bounded mbarrier wait.

#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "attention.cuh"

namespace ckv {

namespace {

constexpr int kTile = 64;
constexpr int kStages = 4;
constexpr int kThreadsAttn = 320;
constexpr uint32_t kEBytes = kTile * 256 * 2;         // 32 KB
constexpr uint32_t kXBytes = 128 * kTile * 4;         // 32 KB
constexpr uint32_t kOffE = 0;
constexpr uint32_t kOffX = kOffE + kStages * kEBytes;
constexpr uint32_t kOffO = 0;                         // final O staging reuses E
constexpr uint32_t kOffML = kOffX + 2 * kXBytes;
constexpr uint32_t kOffBar = kOffML + 128 * 8;
constexpr uint32_t kNumBars = 4 * kStages + 10;
constexpr uint32_t kOffSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffSlot + 16;
constexpr uint32_t kSmemAttn = kSmemUsed + 1024;
static_assert(128 * 256 * 4 <= kOffX, "O staging fits in the E ring");
static_assert(kSmemAttn <= 232448, "fits the 227 KB opt-in limit");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384;
constexpr uint32_t kIdescQK = idesc_bf16(128, kTile, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, 0, 1);
constexpr float kRescaleLog2 = 8.0f;   // lazy rescale threshold (factor 256)

// barrier indices
constexpr int B_TMA = 0, B_EFULL = kStages, B_EEMPTY = 2 * kStages;
constexpr int B_SFULL = 3 * kStages, B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2,
              B_XFULL = B_ODONE + 1, B_CLUSTER = B_XFULL + 2;

// Cluster-wide barrier `k` built on mbarriers with a bounded wait: thread 0
// of every CTA arrives (release, cluster scope) on barrier k of every CTA of
// the cluster after a CTA barrier; every thread then waits on its own CTA's
// barrier k (acquire, cluster scope).  Each barrier is used once (phase 0).
__device__ __forceinline__ void cluster_barrier(uint64_t* bars_k, int n_cta, DevStatus* st,
                                                volatile int* abort, int where) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t local = smem_u32(bars_k);
    for (int r = 0; r < n_cta; ++r) mbar_arrive_remote(mapa(local, (uint32_t)r));
  }
  mbar_wait_poll(bars_k, 0, st, abort, where);
}

// D(tmem) (+)= A(tmem) * B(smem desc), kind::f16.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte chunk `c8` (0..7) of row `r` of a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(uint32_t tile, int r, int c8) {
  return tile + r * 128 + ((c8 ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Tile {
  int win;     // 0 main entries, 1 window slots
  int start;   // first row of the segment
  int valid;   // rows in [start, start + valid)
};

__device__ __forceinline__ Tile tile_of(int t, int nt_main, int n_sel, int n_win) {
  Tile r;
  if (t < nt_main) {
    r.win = 0;
    r.start = t * kTile;
    r.valid = min(kTile, n_sel - r.start);
  } else {
    r.win = 1;
    r.start = (t - nt_main) * kTile;
    r.valid = min(kTile, n_win - r.start);
  }
  return r;
}

struct RowSrc {
  const uint8_t* data;
  const void* scale;
  int64_t entry;  // global slot (b * cap + pos), or -1 when the row is empty
};

// Dequantise local latent chunk `q` of row `src` (half `half`) into the bf16
// tile `tile` at row `r`.  Writes zeros for an empty row.
__device__ __forceinline__ void fill_chunk(const AttnArgs& a, uint32_t tile, int r, int q,
                                           const RowSrc& src, int half) {
  const bool empty = src.entry < 0;
  if (a.fmt == CKV_FMT_BF16) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (!empty) v = *reinterpret_cast<const uint4*>(src.data + src.entry * 1024 + half * 512 + q * 16);
    const int d0 = q * 8;
    st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, (d0 & 63) >> 3), v);
  } else if (a.fmt == CKV_FMT_MIXED) {
    const int n_fp8 = half == 0 ? 16 : 12;
    if (q < n_fp8) {
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
      if (!empty) {
        const uint4 raw = *reinterpret_cast<const uint4*>(src.data + src.entry * 576 + half * 256 + q * 16);
        const int nblk = 448 / a.nope_block;
        const float s = reinterpret_cast<const float*>(src.scale)[src.entry * nblk + (half * 256 + q * 16) / a.nope_block];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __half2_raw h0 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFF), __NV_E4M3);
          __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
          float2 f0 = __half22float2(__half2(h0)), f1 = __half22float2(__half2(h1));
          o[2 * i] = pack_bf16(f0.x * s, f0.y * s);
          o[2 * i + 1] = pack_bf16(f1.x * s, f1.y * s);
        }
        v0 = make_uint4(o[0], o[1], o[2], o[3]);
        v1 = make_uint4(o[4], o[5], o[6], o[7]);
      }
      const int d0 = q * 16;
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, (d0 & 63) >> 3), v0);
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, ((d0 & 63) >> 3) + 1), v1);
    } else {  // rope dims 448..511 (half 1 only), bf16
      const int k = q - 12;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (!empty) v = *reinterpret_cast<const uint4*>(src.data + src.entry * 576 + 448 + k * 16);
      const int d0 = 192 + k * 8;
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, (d0 & 63) >> 3), v);
    }
  } else {  // CKV_FMT_FP4: 8 chunks of 32 channels
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = 0;
    if (!empty) {
      const uint4 raw = *reinterpret_cast<const uint4*>(src.data + src.entry * 256 + half * 128 + q * 16);
      const uint8_t* sp = reinterpret_cast<const uint8_t*>(src.scale) + src.entry * 32 + half * 16 + q * 2;
      const float s0 = e4m3_value(sp[0]), s1 = e4m3_value(sp[1]);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float s = i < 2 ? s0 : s1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t byte = (w[i] >> (8 * k)) & 0xFF;
          o[4 * i + k] = pack_bf16(e2m1_value(byte & 0xF) * s, e2m1_value(byte >> 4) * s);
        }
      }
    }
    const int d0 = q * 32;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, ((d0 & 63) >> 3) + k),
                   make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]));
  }
}

__device__ __forceinline__ int chunks_per_row(int fmt, int half) {
  return fmt == CKV_FMT_BF16 ? 32 : fmt == CKV_FMT_MIXED ? (half == 0 ? 16 : 20) : 8;
}

}  // namespace

__global__ void __launch_bounds__(kThreadsAttn, 1)
    attn_kernel(const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_win,
                const __grid_constant__ AttnBatch batch) {
  const AttnArgs& a = batch.layer[blockIdx.z];
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(gbase + kOffSlot);
  float2* ml = reinterpret_cast<float2*>(gbase + kOffML);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)(rank >> 1), half = (int)(rank & 1);
  const uint32_t peer = rank ^ 1u;
  const int b = blockIdx.y;
  const int G = a.G;
  const bool use_tma = a.use_tma != 0;

  const int n_sel = a.idx ? a.topk : max(0, min(a.n_comp[b], a.n_comp_max));
  const int n_win = max(0, min(a.win_len[b], (int)a.win_cap));
  const int nt_main = (n_sel + kTile - 1) / kTile;
  const int n_tiles = nt_main + (n_win + kTile - 1) / kTile;
  const int t0 = (int)((int64_t)pair * n_tiles / G), t1 = (int)((int64_t)(pair + 1) * n_tiles / G);
  const int n_my = t1 - t0;
  const int32_t* idx_b = a.idx ? a.idx + (int64_t)b * a.topk : nullptr;

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_TMA + s], 1);
      mbar_init(&bars[B_EFULL + s], 128);
      mbar_init(&bars[B_EEMPTY + s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars[B_SFULL + k], 1);
      mbar_init(&bars[B_PFULL + k], 128);
      mbar_init(&bars[B_XFULL + k], 128);
    }
    mbar_init(&bars[B_ODONE], 1);
    mbar_init(&bars[B_CLUSTER], 2 * G);
    mbar_init(&bars[B_CLUSTER + 1], 2 * G);
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(tslot, kTmemCols);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  volatile int* abort_p = &abort_flag;
  const bool prog = a.progress != 0;
  if (tid == 0) progress(a.st, prog, 0);

  if (warp >= 6) {
    // Q[b, h, half] -> TMEM as the bf16 A operand (lane h, two elements per column)
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      if (h < a.H) {
        const uint4* src = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.H + h) * 512 + half * 256 + c * 64);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = src[k];
          r[4 * k] = v.x;
          r[4 * k + 1] = v.y;
          r[4 * k + 2] = v.z;
          r[4 * k + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
      tmem_st32(tmem + lane_base + kColQ + c * 32, r);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    // ------------------------------------------------------ TMA issuer ----
    if (use_tma && lane == 0) {
      for (int i = 0; i < n_my; ++i) {
        const int s = i % kStages;
        if (i >= kStages &&
            !mbar_wait(&bars[B_EEMPTY + s], ((i / kStages) + 1) & 1, a.st, abort_p, 21))
          break;
        const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
        const CUtensorMap* map = tl.win ? &map_win : &map_kv;
        const int64_t row = (int64_t)b * (tl.win ? a.win_cap : a.kv_cap) + tl.start;
        progress(a.st, prog, 9);
        mbar_expect_tx(&bars[B_TMA + s], kEBytes);
#pragma unroll
        for (int kc = 0; kc < 4; ++kc)
          tma_load_2d(base + kOffE + s * kEBytes + kc * 8192, map, half * 256 + kc * 64, (int)row,
                      &bars[B_TMA + s]);
      }
    }
    __syncwarp();
  } else if (warp >= 1 && warp <= 4) {
    // ------------------------------------------- producers / TMA fix-up ----
    const int p = tid - 32;
    const int J = chunks_per_row(a.fmt, half);
    for (int i = 0; i < n_my; ++i) {
      const int s = i % kStages;
      const uint32_t tile = base + kOffE + s * kEBytes;
      const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
      if (use_tma) {
        if (!mbar_wait(&bars[B_TMA + s], (i / kStages) & 1, a.st, abort_p, 22)) break;
        if (tl.valid < kTile) {
          // rows past the end of the segment: zero them so that P = 0 meets
          // finite values in P.E
          for (int j = p; j < (kTile - tl.valid) * 32; j += 128) {
            const int r = tl.valid + (j >> 5), cc = j & 31;
            st_shared_v4(sw128(tile + (cc >> 3) * 8192, r, cc & 7), make_uint4(0, 0, 0, 0));
          }
        }
      } else {
        if (i >= kStages &&
            !mbar_wait(&bars[B_EEMPTY + s], ((i / kStages) + 1) & 1, a.st, abort_p, 23))
          break;
        for (int j = p; j < kTile * J; j += 128) {
          const int r = j / J, q = j - r * J;
          RowSrc src;
          src.entry = -1;
          if (r < tl.valid) {
            const int row = tl.start + r;
            if (!tl.win) {
              int64_t e = idx_b ? (int64_t)__ldg(idx_b + row) : row;
              if (e >= a.kv_cap) {
                if (q == 0 && half == 0) report(a.st, CKV_ERR_DEVICE_BOUNDS, (int)e);
                e = -1;
              }
              if (e >= 0) {
                src.data = a.kv_data;
                src.scale = a.kv_scale;
                src.entry = (int64_t)b * a.kv_cap + e;
              }
            } else {
              src.data = a.win_data;
              src.scale = a.win_scale;
              src.entry = (int64_t)b * a.win_cap + row;
            }
          }
          fill_chunk(a, tile, r, q, src, half);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[B_EFULL + s]);
      if (p == 0) progress(a.st, prog, 5);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      const uint32_t tO = tmem + kColO, tQ = tmem + kColQ;
      auto issue_pv = [&](int j) -> bool {
        const int sj = j % kStages, bj = j & 1;
        if (!mbar_wait(&bars[B_PFULL + bj], (j >> 1) & 1, a.st, abort_p, 24)) return false;
        tc_fence_after();
        const uint32_t tile = base + kOffE + sj * kEBytes;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t db = smem_desc(tile + ks * 2048, 8192, 1024, 2);
          umma_f16_ta(tO, tmem + kColS + 64 * bj + 8 * ks, db, kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_ODONE]);
        umma_commit(&bars[B_EEMPTY + sj]);
        progress(a.st, prog, 4);
        return true;
      };
      bool ok = true;
      for (int i = 0; i < n_my && ok; ++i) {
        const int s = i % kStages, bi = i & 1;
        const uint32_t tile = base + kOffE + s * kEBytes;
        if (!mbar_wait(&bars[B_EFULL + s], (i / kStages) & 1, a.st, abort_p, 25)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint32_t kc = ks >> 2, w = ks & 3;
          const uint64_t db = smem_desc(tile + kc * 8192 + w * 32, 16, 1024, 2);
          umma_f16_ta(tmem + kColS + 64 * bi, tQ + 8 * ks, db, kIdescQK, ks > 0);
        }
        umma_commit(&bars[B_SFULL + bi]);
        progress(a.st, prog, 1);
        if (i > 0) ok = issue_pv(i - 1);
      }
      if (ok && n_my > 0) issue_pv(n_my - 1);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax (row = head) ----
    const int qd = warp & 3;
    const int h = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t tO = tmem + kColO + lane_base;
    float m_used = -INFINITY, l = 0.f;
    for (int i = 0; i < n_my; ++i) {
      const int bi = i & 1;
      const uint32_t tS = tmem + kColS + 64 * bi + lane_base;
      if (!mbar_wait(&bars[B_SFULL + bi], (i >> 1) & 1, a.st, abort_p, 26)) break;
      tc_fence_after();
      if (h == 0) progress(a.st, prog, 2);
      uint32_t sr[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld();
      // swap the partial scores with the other half of the pair
      const uint32_t xrow = base + kOffX + bi * kXBytes + h * 256;
      const uint32_t xrow_peer = mapa(xrow, peer);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_cluster_v4(xrow_peer + ((c ^ (h & 7)) << 4),
                      make_float4(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1]),
                                  __uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3])));
      mbar_arrive_remote(mapa(smem_u32(&bars[B_XFULL + bi]), peer));
      const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
      // validity of the tile's rows (selected entries may be -1 / out of range)
      uint64_t vmask = tl.valid >= 64 ? ~0ull : ((1ull << tl.valid) - 1ull);
      if (!tl.win && idx_b) {
        uint64_t im = 0;
        for (int j = 0; j < tl.valid; ++j) {
          const int e = __ldg(idx_b + tl.start + j);
          im |= (uint64_t)(e >= 0 && e < a.kv_cap) << j;
        }
        vmask &= im;
      }
      if (!mbar_wait_poll(&bars[B_XFULL + bi], (i >> 1) & 1, a.st, abort_p, 27)) break;
      if (h == 0) progress(a.st, prog, 3);
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float4 o = ld_shared_v4f(xrow + ((c ^ (h & 7)) << 4));
        const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = 4 * c + k;
          const float z = ((vmask >> j) & 1ull) ? (__uint_as_float(sr[j]) + ov[k]) * a.scale_log2 : -INFINITY;
          sr[j] = __float_as_uint(z);
          tmax = fmaxf(tmax, z);
        }
      }
      if (tmax > m_used + kRescaleLog2 || (m_used == -INFINITY && tmax > -INFINITY)) {
        const float m_new = tmax;
        if (i > 0 && m_used != -INFINITY) {
          // PV(i-1) must be done before O is rescaled
          if (!mbar_wait(&bars[B_ODONE], (i - 1) & 1, a.st, abort_p, 28)) break;
          tc_fence_after();
          const float alpha = fast_exp2(m_used - m_new);
          l *= alpha;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            tmem_ld32(tO + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
            tmem_st32(tO + c * 32, r);
          }
          tmem_wait_st();
        }
        m_used = m_new;
      }
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float z0 = __uint_as_float(sr[2 * k]), z1 = __uint_as_float(sr[2 * k + 1]);
        const float p0 = m_used == -INFINITY ? 0.f : fast_exp2(z0 - m_used);
        const float p1 = m_used == -INFINITY ? 0.f : fast_exp2(z1 - m_used);
        __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        const float2 pr = __bfloat1622float2(pb);
        l += pr.x + pr.y;
        pk[k] = *reinterpret_cast<uint32_t*>(&pb);
      }
      tmem_st32(tS, pk);   // P over the first 32 columns of this S buffer
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[B_PFULL + bi]);
      if (h == 0) progress(a.st, prog, 8);
    }
    if (n_my > 0) {
      // s_full of the last tile implies every PV up to n_my - 3 is done, so
      // o_done may still owe two phases: wait for them in order (a single
      // parity wait could alias the older one).
      if (n_my >= 2) mbar_wait(&bars[B_ODONE], (n_my - 2) & 1, a.st, abort_p, 29);
      mbar_wait(&bars[B_ODONE], (n_my - 1) & 1, a.st, abort_p, 29);
      tc_fence_after();
    }
    // stage this CTA's partial accumulator for the in-cluster merge
    const uint32_t orow = base + kOffO + h * 1024;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t r[32];
      if (n_my > 0) {
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c4 = c * 8 + k;
        st_shared_v4(orow + (((c4 & ~7) | ((c4 & 7) ^ (h & 7))) << 4),
                     make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]));
      }
    }
    ml[h] = make_float2(m_used, l);
  }
  tc_fence_before();
  if (tid == 0) progress(a.st, prog, 6);
  cluster_barrier(&bars[B_CLUSTER], 2 * G, a.st, abort_p, 30);

  if (warp >= 6) {
    // --------------------------------------------- in-cluster merge ----
    const int h = (warp & 3) * 32 + lane;
    float mq[4] = {0.f, 0.f, 0.f, 0.f}, wq[4] = {0.f, 0.f, 0.f, 0.f};
    float M = -INFINITY;
    for (int q = 0; q < G; ++q) {
      const uint32_t rq = 2u * q + half;
      mq[q] = ld_cluster_f32(mapa(smem_u32(&ml[h].x), rq));
      wq[q] = ld_cluster_f32(mapa(smem_u32(&ml[h].y), rq));
      M = fmaxf(M, mq[q]);
    }
    float L = 0.f;
    for (int q = 0; q < G; ++q) {
      const float f = mq[q] == -INFINITY ? 0.f : exp2f(mq[q] - M);
      L += wq[q] * f;
      mq[q] = f;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int cols = 256 / G, c4_0 = pair * cols / 4;
    if (h < a.H) {
      __nv_bfloat16* out = a.out + ((int64_t)b * a.H + h) * 512 + half * 256;
      const uint32_t orow = base + kOffO + h * 1024;
      uint32_t rbase[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) rbase[q] = mapa(orow, 2u * (q < G ? q : 0) + half);
      for (int c4 = c4_0; c4 < c4_0 + cols / 4; c4 += 2) {
        // issue every partial's loads first, then accumulate
        float4 v[4][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int cc = c4 + u;
            v[q][u] = (q < G && mq[q] != 0.f)
                          ? ld_cluster_v4(rbase[q] + (((cc & ~7) | ((cc & 7) ^ (h & 7))) << 4))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float f = q < G ? mq[q] : 0.f;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            acc[4 * u] += f * v[q][u].x;
            acc[4 * u + 1] += f * v[q][u].y;
            acc[4 * u + 2] += f * v[q][u].z;
            acc[4 * u + 3] += f * v[q][u].w;
          }
        }
        uint4 o;
        o.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        o.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        o.z = pack_bf16(acc[4] * inv, acc[5] * inv);
        o.w = pack_bf16(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(out + c4 * 4) = o;
      }
      if (rank == 0 && a.lse)
        a.lse[(int64_t)b * a.H + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  cluster_barrier(&bars[B_CLUSTER + 1], 2 * G, a.st, abort_p, 31);
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0) progress(a.st, prog, 7);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_attn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over a BF16 plane viewed as [rows][512] bf16, box 64 x 64, 128B swizzle.
bool encode_bf16_rows(CUtensorMap* m, const void* data, int64_t rows) {
  auto enc = encode_fn_attn();
  if (!enc || rows <= 0 || rows >= ((int64_t)1 << 31)) return false;
  cuuint64_t dims[2] = {512, (cuuint64_t)rows};
  cuuint64_t strides[1] = {1024};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(data), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attention_layers(const AttnArgs* layers, int n, int B, cudaStream_t stream) {
  static int attr_done = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_done != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemAttn);
    if (e != cudaSuccess) return e;
    attr_done = dev;
  }
  if (n < 1 || n > kMaxLayers) return cudaErrorInvalidValue;
  AttnBatch batch;
  memset(&batch, 0, sizeof(batch));
  for (int l = 0; l < n; ++l) {
    batch.layer[l] = layers[l];
    batch.layer[l].use_tma = 0;
  }
  CUtensorMap mk, mw;
  memset(&mk, 0, sizeof(mk));
  memset(&mw, 0, sizeof(mw));
  // Contiguous BF16 rows (HCA, one layer) stream through TMA; gathered or
  // quantised rows go through the producer warps.
  const AttnArgs& a0 = layers[0];
  if (n == 1 && a0.fmt == CKV_FMT_BF16 && a0.idx == nullptr &&
      encode_bf16_rows(&mk, a0.kv_data, (int64_t)B * a0.kv_cap) &&
      encode_bf16_rows(&mw, a0.win_data, (int64_t)B * a0.win_cap))
    batch.layer[0].use_tma = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a0.G, B, n);
  cfg.blockDim = dim3(kThreadsAttn, 1, 1);
  cfg.dynamicSmemBytes = kSmemAttn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * a0.G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_kernel, mk, mw, batch);
}

cudaError_t launch_attention(const AttnArgs& a, int B, cudaStream_t stream) {
  return launch_attention_layers(&a, 1, B, stream);
}

}  // namespace ckv

// csa_sparse_attn / hca_attn: shared-KV decode attention on tcgen05.
//
// "DeepSeek-V4 KV Cache 深度分析": §五 -- each compressed entry is both key
// and value (o = sum_j a_j C_j); §十一 -- Attention(Q, selected) followed by
// the 128-token window; §三 -- HCA attends densely to every ratio-128 entry
// plus the window.  One softmax over the union of the rows (no sink).
//
// Decomposition (per sequence b, 2G CTAs: G pairs; a cluster is either all
// 2G CTAs of the sequence or one pair, whichever lets more pairs run):
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
//   * The G pairs merge (m, l, O) at the end through the workspace: every CTA
//     writes its partial (O / l in fp16, (m, l) in f32; it stays in L2), the
//     sequence's CTAs meet (the cluster barrier, or with pair clusters a
//     bounded counter in the workspace), and CTA (p, c) finalises latent
//     columns [256c + p*256/G, ...) from the G partials of half c.
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
#include "tmap.cuh"

namespace ckv {

namespace {

constexpr int kTile = 64;
constexpr int kStages = 5;
constexpr int kThreadsAttn = 320;
constexpr uint32_t kEBytes = kTile * 256 * 2;         // 32 KB
constexpr uint32_t kXBytes = 128 * kTile * 2;         // 16 KB: fp16 partial scores
constexpr uint32_t kOffE = 0;
constexpr uint32_t kOffX = kOffE + kStages * kEBytes;
constexpr int kXBufs = 4;                              // send-ahead needs four
constexpr uint32_t kOffRowSrc = kOffX + kXBufs * kXBytes;    // int32 [kStages][64]
constexpr uint32_t kOffVmask = kOffRowSrc + kStages * 64 * 4;  // u32 [kStages][2]
// Raw bytes of a gathered tile, staged inside its own 32 KB stage buffer
// before they are dequantised over it: MIXED rows (256 or 320 bytes) from
// byte 8192 and each row's f32 scale words (32 bytes a row) from 28672; FP4
// rows (128 bytes) from byte 16384 and their 16 scale bytes from 24576, in
// 128-byte groups of four rows (every TMA destination is 128-byte aligned).
constexpr uint32_t kRawOffMixed = 8192, kScaleOffMixed = 28672;
constexpr uint32_t kRawOffFp4 = 16384, kScaleOffFp4 = 24576;
static_assert(kRawOffMixed + 64 * 320 <= kScaleOffMixed && kScaleOffMixed + 64 * 32 <= kEBytes,
              "MIXED staging fits in a stage");
static_assert(kRawOffFp4 + 64 * 128 <= kScaleOffFp4 && kScaleOffFp4 + 16 * 128 <= kEBytes,
              "FP4 staging fits in a stage");
constexpr uint32_t kOffBar = kOffVmask + kStages * 8;
constexpr uint32_t kNumBars = 5 * kStages + 12;
constexpr uint32_t kOffSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffRope = kOffSlot + 16;                 // float2 [32]: (cos, sin) of rope pair k
constexpr uint32_t kSmemUsed = kOffRope + 32 * 8;
constexpr uint32_t kSmemAttn = kSmemUsed + 1024;
static_assert(kSmemAttn <= 232448, "fits the 227 KB opt-in limit");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384;
constexpr uint32_t kIdescQK = idesc_bf16(128, kTile, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, 0, 1);
constexpr float kRescaleLog2 = 8.0f;   // lazy rescale threshold (factor 256)

// barrier indices
constexpr int B_TMA = 0, B_EFULL = kStages, B_EEMPTY = 2 * kStages;
constexpr int B_SFULL = 3 * kStages, B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2,
              B_XFULL = B_ODONE + 1, B_CLUSTER = B_XFULL + kXBufs, B_XREAD = B_CLUSTER + 2,
              B_GFULL = B_XREAD + 2;
static_assert(B_GFULL + kStages <= (int)kNumBars, "barrier count");

// Cluster-wide barrier `k` built on mbarriers with a bounded wait: after a
// CTA barrier, thread r of every CTA arrives (release, cluster scope, which
// also covers the writes the CTA barrier ordered before it) on barrier k of
// CTA r, all CTAs in parallel; every thread then waits on its own CTA's
// barrier k (acquire, cluster scope).  Each barrier is used once (phase 0).
__device__ __forceinline__ void cluster_barrier(uint64_t* bars_k, int n_cta, DevStatus* st,
                                                volatile int* abort, int where) {
  __syncthreads();
  if ((int)threadIdx.x < n_cta) mbar_arrive_remote(mapa(smem_u32(bars_k), threadIdx.x));
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

// Fetch a tensor map's descriptor ahead of its first use.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Four rows (y0..y3; a negative or out-of-range row reads zeros) of the
// one-row box at column x of a 2-D tensor map, stacked at dst.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0,
                                            int y1, int y2, int y3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
      "r"(smem_u32(bar))
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

constexpr int64_t kPart16 = 2 * kPartFloats / 4;   // 16-byte stride between pairs' partials

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

// Asynchronous 4-byte global -> shared copies (cp.async) for the MIXED
// scale words (the 16-byte chunks of gathered quantised rows use cp_async16).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most `n` (0..3) of this thread's newest copy groups are pending.
__device__ __forceinline__ void cp_async_wait(int n) {
  if (n <= 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
  else if (n == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
  else if (n == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
  else asm volatile("cp.async.wait_group 3;" ::: "memory");
}
// Named barrier `id` over `n` threads that also ANDs `v` across them, so a
// failed wait in any thread makes every thread leave the loop together.
__device__ __forceinline__ bool bar_and(int id, int n, bool v) {
  int r;
  asm volatile(
      "{\n .reg .pred pv, pr;\n setp.ne.b32 pv, %1, 0;\n bar.red.and.pred pr, %2, %3, pv;\n"
      " selp.b32 %0, 1, 0, pr;\n}\n"
      : "=r"(r)
      : "r"((int)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Raw bytes of one 16-byte source chunk of a row plus its scale bits.
struct Raw {
  uint4 v;
  uint32_t s;   // MIXED: f32 scale bits; FP4: two E4M3 scale bytes
};

// Dequantise a loaded chunk to bf16 and store it at row `r` of the swizzled
// tile (an empty row stores zeros: its raw bytes and scale are zero).  Out of
// line, the chunk passed in registers: the producers' unrolled chunk loop
// then holds one copy of the conversion, which matters when the kernel starts
// with its code evicted from the instruction caches (in a decode step the
// index kernel runs just before): 2 us less per step at 128 k and 1 M.
template <int FMT>
__device__ __noinline__ void store_chunk(const AttnArgs& a, uint32_t tile, int r, int q,
                                        const Raw raw, int half) {
  if constexpr (FMT == CKV_FMT_BF16) {
    const int d0 = q * 8;
    st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, (d0 & 63) >> 3), raw.v);
  } else if constexpr (FMT == CKV_FMT_MIXED) {
    const int n_fp8 = half == 0 ? 16 : 12;
    if (q < n_fp8) {
      const float s = __uint_as_float(raw.s);
      const uint32_t w[4] = {raw.v.x, raw.v.y, raw.v.z, raw.v.w};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __half2_raw h0 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFF), __NV_E4M3);
        __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
        float2 f0 = __half22float2(__half2(h0)), f1 = __half22float2(__half2(h1));
        o[2 * i] = pack_bf16(f0.x * s, f0.y * s);
        o[2 * i + 1] = pack_bf16(f1.x * s, f1.y * s);
      }
      const int d0 = q * 16;
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, (d0 & 63) >> 3), make_uint4(o[0], o[1], o[2], o[3]));
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, ((d0 & 63) >> 3) + 1), make_uint4(o[4], o[5], o[6], o[7]));
    } else {  // rope dims 448..511 (half 1 only), bf16
      const int d0 = 192 + (q - 12) * 8;
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, (d0 & 63) >> 3), raw.v);
    }
  } else {  // FP4: 32 channels
    // Hardware conversions: two E2M1 codes -> f16x2, the E4M3 scale -> f16;
    // a code times a scale has at most 6 significant bits and stays within
    // f16's range, so the f16 product and its BF16 rounding are exact.
    const __half2 s0 = __half2half2(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(raw.s & 0xFF), __NV_E4M3)));
    const __half2 s1 = __half2half2(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(raw.s >> 8), __NV_E4M3)));
    const uint32_t w[4] = {raw.v.x, raw.v.y, raw.v.z, raw.v.w};
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 sc = i < 2 ? s0 : s1;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // low nibble = even channel = .x
        const __half2 hv = __hmul2(__half2(__nv_cvt_fp4x2_to_halfraw2(
                                       (__nv_fp4x2_storage_t)((w[i] >> (8 * k)) & 0xFF), __NV_E2M1)),
                                   sc);
        const float2 f = __half22float2(hv);
        o[4 * i + k] = pack_bf16(f.x, f.y);
      }
    }
    const int d0 = q * 32;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      st_shared_v4(sw128(tile + (d0 >> 6) * 8192, r, ((d0 & 63) >> 3) + k),
                   make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]));
  }
}

template <int FMT>
__device__ __forceinline__ int chunks_per_row(int half) {
  return FMT == CKV_FMT_BF16 ? 32 : FMT == CKV_FMT_MIXED ? (half == 0 ? 16 : 20) : 8;
}

// j / J for the chunk counts above, with constant divisors.
template <int FMT>
__device__ __forceinline__ int chunk_row(int j, int half) {
  if constexpr (FMT == CKV_FMT_BF16) return j >> 5;
  else if constexpr (FMT == CKV_FMT_MIXED) return half == 0 ? (j >> 4) : j / 20;
  else return j >> 3;
}

}  // namespace

namespace {

// Combines the G partials of one half over units [u0, u1) of 8 columns x H
// head rows into `out`, staged through shared memory at `stage` (room for
// kMergeStagePieces 16-byte pieces): per pass, every piece of P items x G
// partials is copied by cp.async, all in flight at once, while warps 6..9
// turn each row's (m, l) of the G pairs into the weights l_q 2^(m_q - M) / L
// (`wsm`, 2 x kMaxPairs x 128 floats; the first pass only) and, when lse is
// not null, write its log-sum-exp; then each thread forms its items from
// shared memory, one partial at a time.  Out of line and rolled over the partials: the merge
// runs once per call, usually with its code cold in the instruction caches.
//
// rtab (null: none): (cos, sin) of the 32 rope pairs; the units holding the
// last 64 latent dims (units 24..31 of half 1) are turned by the opposite
// angle before they are stored (the output's RoPE at position -i).
constexpr uint32_t kMergeWBytes = 2 * kMaxPairs * 128 * 4;
constexpr int kMergeStagePieces = (int)((kStages * kEBytes - kMergeWBytes) / 16);

__device__ __noinline__ void merge_partials(const uint4* pq0, float* wsm, uint32_t stage, int G, int H,
                                            __nv_bfloat16* out, float* lse, int tid, int u0, int u1,
                                            const float2* rtab) {
  const int n_items = (u1 - u0) * H;   // only the H real head rows
  const int P = kMergeStagePieces / G;
  const int warp = tid >> 5, lane = tid & 31;
#pragma unroll 1
  for (int p0 = 0; p0 < n_items; p0 += P) {
    const int np = min(P, n_items - p0);
    // item k of the pass is row hh of unit uu: (uu, hh) advance with k
    const int kf = p0 + tid, uf = u0 + kf / H, hf = kf - (uf - u0) * H;
    auto step = [&](int& uu, int& hh) {
      hh += kThreadsAttn;
#pragma unroll 1
      while (hh >= H) {
        hh -= H;
        ++uu;
      }
    };
    int uu = uf, hh = hf;
#pragma unroll 1
    for (int k = tid; k < np; k += kThreadsAttn, step(uu, hh)) {
      const uint4* src = pq0 + uu * 128 + hh;
#pragma unroll 1
      for (int q = 0; q < G; ++q) cp_async16(stage + (uint32_t)(q * P + k) * 16u, src + q * kPart16);
    }
    cp_async_commit();
    if (p0 == 0 && warp >= 6) {
      const int h = (warp & 3) * 32 + lane;
      float M = -INFINITY;
      float2 ml[kMaxPairs];   // every pair's (m, l) load in flight at once
#pragma unroll
      for (int q = 0; q < kMaxPairs; ++q)
        ml[q] = q < G ? __ldcg(reinterpret_cast<const float2*>(pq0 + q * kPart16 + 32 * 128) + h)
                      : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int q = 0; q < kMaxPairs; ++q) {
        wsm[q * 128 + h] = ml[q].x;   // m_q (the weight from the next loop on)
        wsm[(kMaxPairs + q) * 128 + h] = ml[q].y;
        M = fmaxf(M, ml[q].x);
      }
      float L = 0.f;
#pragma unroll 1
      for (int q = 0; q < G; ++q) {
        const float mq = wsm[q * 128 + h], lq0 = wsm[(kMaxPairs + q) * 128 + h];
        const float lq = mq == -INFINITY ? 0.f : lq0 * exp2f(mq - M);
        wsm[q * 128 + h] = lq;
        L += lq;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll 1
      for (int q = 0; q < G; ++q) wsm[q * 128 + h] *= inv;
      if (lse && h < H) lse[h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    uu = uf;
    hh = hf;
#pragma unroll 1
    for (int k = tid; k < np; k += kThreadsAttn, step(uu, hh)) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      // two partials per step: their loads in flight together
#pragma unroll 1
      for (int q = 0; q < G; q += 2) {
        const bool two = q + 1 < G;
        const float w0 = wsm[q * 128 + hh], w1 = two ? wsm[(q + 1) * 128 + hh] : 0.f;
        const uint4 v0 = ld_shared_u4(stage + (uint32_t)(q * P + k) * 16u);
        const uint4 v1 = two ? ld_shared_u4(stage + (uint32_t)((q + 1) * P + k) * 16u) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t x0[4] = {v0.x, v0.y, v0.z, v0.w}, x1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&x0[e]));
          acc[2 * e] += w0 * f.x;
          acc[2 * e + 1] += w0 * f.y;
        }
        if (two) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&x1[e]));
            acc[2 * e] += w1 * f.x;
            acc[2 * e + 1] += w1 * f.y;
          }
        }
      }
      if (rtab && uu >= 24) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 cs = rtab[4 * (uu - 24) + e];
          const float re = acc[2 * e], im = acc[2 * e + 1];
          acc[2 * e] = re * cs.x + im * cs.y;
          acc[2 * e + 1] = im * cs.x - re * cs.y;
        }
      }
      uint4 o;
      o.x = pack_bf16(acc[0], acc[1]);
      o.y = pack_bf16(acc[2], acc[3]);
      o.z = pack_bf16(acc[4], acc[5]);
      o.w = pack_bf16(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(out + (int64_t)hh * 512 + 8 * uu) = o;
    }
    __syncthreads();   // the staging area is written again by the next pass
  }
}


}  // namespace

// Debug timeline (progress mode 2 / 4): CTA (0 / 1, 0, 0) stores clock64 offsets of
// its pipeline hand-offs in the status block's spare words.
static __device__ __noinline__ void trace_store(DevStatus* st, int slot, long long t0) {
  if (slot < 61) st->pad[slot] = (int32_t)(clock64() - t0);
}
__device__ __forceinline__ void trace(DevStatus* st, bool on, int slot, long long t0) {
  if (on) trace_store(st, slot, t0);
}

template <int FMT>
__global__ void __launch_bounds__(kThreadsAttn, 1)
    attn_kernel(const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_win,
                const __grid_constant__ AttnBatch batch) {
  const AttnArgs& a = batch.layer[blockIdx.z];
  if (a.tag != (kArgsTag ^ (int)blockIdx.z)) {
    // a damaged argument block: touch none of its pointers (every CTA of
    // the cluster takes this branch, so none waits on the others).  The CTA
    // still waits for the previous grid before it leaves: a grid whose CTAs
    // all left without waiting could complete before its predecessor and
    // release the next launch of the stream too early.
    pdl_wait();
    if (threadIdx.x == 0) report(batch.layer[0].st, CKV_ERR_INVALID, (int)blockIdx.z);
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(gbase + kOffSlot);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A cluster is either one pair or all 2G CTAs of the sequence
  // (a.cluster_all); either way CTA x of the sequence is pair x / 2, half
  // x % 2, and its peer is the adjacent cluster rank.
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)(blockIdx.x >> 1), half = (int)(blockIdx.x & 1);
  const uint32_t peer = rank ^ 1u;
  const int b = blockIdx.y;
  const int G = a.G;
  const bool use_tma = FMT == CKV_FMT_BF16 && a.use_tma != 0;   // contiguous BF16 rows only

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
    }
    for (int k = 0; k < kXBufs; ++k) mbar_init(&bars[B_XFULL + k], 128);
    mbar_init(&bars[B_XREAD], 128);
    mbar_init(&bars[B_XREAD + 1], 128);
    for (int k = 0; k < kStages; ++k) mbar_init(&bars[B_GFULL + k], 1);
    mbar_init(&bars[B_ODONE], 1);
    mbar_init(&bars[B_CLUSTER], a.cluster_all ? 2 * a.G : 2);
    mbar_init(&bars[B_CLUSTER + 1], a.cluster_all ? 2 * a.G : 2);
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(tslot, kTmemCols);
  if (tid == 32) {
    // kernel parameters, not outputs of the previous kernel: fetched
    // before the grid dependency resolves
    if (use_tma) {
      prefetch_tmap(&map_kv);
      prefetch_tmap(&map_win);
    } else if (FMT == CKV_FMT_BF16) {
      for (int k = 0; k < 4; ++k) prefetch_tmap(&a.gmap[k]);
    }
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // Everything above touches only this CTA's own resources; global memory
  // (inputs included) only after the previous kernel in the stream is done.
  pdl_wait();
  const int n_sel = a.idx ? a.topk : max(0, min(a.n_comp[b], a.n_comp_max));
  const int n_win = max(0, min(a.win_len[b], (int)a.win_cap));
  const int nt_main = (n_sel + kTile - 1) / kTile;
  const int n_tiles = nt_main + (n_win + kTile - 1) / kTile;
  const int t0 = (int)((int64_t)pair * n_tiles / G), t1 = (int)((int64_t)(pair + 1) * n_tiles / G);
  const int n_my = t1 - t0;
  const int32_t* idx_b = a.idx ? a.idx + (int64_t)b * a.topk : nullptr;

  volatile int* abort_p = &abort_flag;
  const bool prog = a.progress == 1;
  // progress modes 2 / 4 trace CTA 0 / 1 of sequence 0 over tiles 0..7,
  // modes 5 / 6 the same CTAs over tiles 8..15
  const bool tr = (a.progress == 2 || a.progress >= 4) && blockIdx.y == 0 && blockIdx.z == 0 &&
                  (int)blockIdx.x == ((a.progress == 4 || a.progress == 6) ? 1 : 0);
  const int toff = a.progress >= 5 ? 8 : 0;
  const long long tr0 = clock64();
  // progress mode 3: the CTAs of sequence 0 (layer 0) store %globaltimer
  // (low 32 bits) at start, softmax end and cluster-barrier exit
  const bool tr3 = a.progress == 3 && blockIdx.y == 0 && blockIdx.z == 0 && blockIdx.x < 12;
  auto stamp3 = [&](int k) {
    if (tr3) a.st->pad[4 * blockIdx.x + k] = (int32_t)(uint32_t)globaltimer();
  };
  if (tid == 0) stamp3(0);
  if (tid == 0) progress(a.st, prog, 0);

  // Rounds this CTA's partial scores S(k) of head row `hq` (TMEM lane
  // quadrant of the calling warp) to fp16 and stores them into the peer's
  // exchange buffer k % kXBufs; the caller arrives on the peer's barrier.
  auto send_scores = [&](int k, int hq) {
    const uint32_t tS = tmem + kColS + 64 * (k & 1) + ((uint32_t)(hq & ~31) << 16);
    const uint32_t xrow_peer = mapa(base + kOffX + (k % kXBufs) * kXBytes + hq * 128, peer);
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t sr[32];
      tmem_ld32(tS + 32 * hh, sr);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t w4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = 8 * i + 2 * u;
          __half2 hv = __floats2half2_rn(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1]));
          w4[u] = *reinterpret_cast<uint32_t*>(&hv);
        }
        st_cluster_u4(xrow_peer + (((4 * hh + i) ^ (hq & 7)) << 4), make_uint4(w4[0], w4[1], w4[2], w4[3]));
      }
    }
  };

  if (warp >= 6) {
    // Q[b, h, half]: the thread's 512 bytes are all requested at once (one
    // memory round trip, however loaded the memory system is).
    const int h = (warp & 3) * 32 + lane;
    uint4 qv[32];
    if (h < a.H) {
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.H + h) * 512 + half * 256);
#pragma unroll
      for (int k = 0; k < 32; ++k) qv[k] = __ldg(src + k);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) qv[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    // RoPE table of this sequence ("DeepSeek-V4 KV Cache 深度分析", §五: the
    // query's and the output's last 64 dims, i.e. half 1): pair k turns by
    // i * theta_k, reduced modulo 2 pi in double precision first.
    const bool rope = half == 1 && a.rope_pos != nullptr && (a.rope_q || a.rope_out);
    float2* rtab = reinterpret_cast<float2*>(gbase + kOffRope);
    if (rope) {
      if (warp == 6) {
        const double ang = (double)a.rope_pos[b] * (double)a.rope_freq[lane];
        const double red = fma(-6.283185307179586, rint(ang * 0.15915494309189535), ang);
        // |red| <= pi: the hardware approximation's absolute error there is
        // about 2^-21, far below the bf16 rounding that follows
        float sv, cv;
        __sincosf((float)red, &sv, &cv);
        rtab[lane] = make_float2(cv, sv);
      }
      asm volatile("bar.sync 4, 128;" ::: "memory");
    }
    // Q -> TMEM as the bf16 A operand (lane h, two elements per column)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        r[4 * k] = qv[8 * c + k].x;
        r[4 * k + 1] = qv[8 * c + k].y;
        r[4 * k + 2] = qv[8 * c + k].z;
        r[4 * k + 3] = qv[8 * c + k].w;
      }
      if (c == 3 && rope && a.rope_q && h < a.H) {
        // dims 448 + 2k, 449 + 2k (one bf16 pair per word) turn by +i theta_k
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 cs = rtab[k];
          const float re = __uint_as_float(r[k] << 16), im = __uint_as_float(r[k] & 0xFFFF0000u);
          r[k] = pack_bf16(re * cs.x - im * cs.y, re * cs.y + im * cs.x);
        }
      }
      tmem_st32(tmem + lane_base + kColQ + c * 32, r);
    }
    tmem_wait_st();
  }
  // Only the MMA and softmax warps need Q in TMEM: the loader warps start
  // fetching the first tiles while Q is being loaded.
  if (warp >= 5) {
    tc_fence_before();
    asm volatile("bar.sync 3, 160;" ::: "memory");
    tc_fence_after();
  }
  if (tid == 0) trace(a.st, tr, 0, tr0);

  if (warp == 0) {
    // ------------------------------------------------------ TMA issuer ----
    // Contiguous BF16 rows by TMA, lane 0 issuing.  With a paged main KV
    // the whole warp fetches the pages of the next 32 tiles (a 64-row tile
    // lies in one page).
    if (use_tma) {
      int pg_reg = 0;
#pragma unroll 1
      for (int i = 0; i < n_my; ++i) {
        const int s = i % kStages;
        bool ok = true;
        if (lane == 0 && i >= kStages)
          ok = mbar_wait(&bars[B_EEMPTY + s], ((i / kStages) + 1) & 1, a.st, abort_p, 21);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
        const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
        int64_t row = (int64_t)b * (tl.win ? a.win_cap : a.kv_cap) + tl.start;
        if (a.kv_bt) {
          if ((i & 31) == 0) {
            const Tile tq = tile_of(t0 + min(i + lane, n_my - 1), nt_main, n_sel, n_win);
            pg_reg = tq.win ? 0 : __ldg(a.kv_bt + (int64_t)b * a.kv_bt_cols + tq.start / a.kv_page);
          }
          const int pg = __shfl_sync(0xffffffffu, pg_reg, i & 31);
          if (!tl.win) row = (int64_t)pg * a.kv_page + tl.start % a.kv_page;
        }
        if (lane == 0) {
          const CUtensorMap* map = tl.win ? &map_win : &map_kv;
          progress(a.st, prog, 9);
          mbar_expect_tx(&bars[B_TMA + s], kEBytes);
#pragma unroll
          for (int kc = 0; kc < 4; ++kc)
            tma_load_2d(base + kOffE + s * kEBytes + kc * 8192, map, half * 256 + kc * 64, (int)row,
                        &bars[B_TMA + s]);
        }
      }
    }
    __syncwarp();
  } else if (warp >= 1 && warp <= 4) {
    // ------------------------------------------- producers / TMA fix-up ----
    const int p = tid - 32;
    const int J = chunks_per_row<FMT>(half);
    if (use_tma) {
      // TMA-fed tiles: these warps release each landed tile to the MMA
      // (zeroing rows past the end of its segment, so that P = 0 meets finite
      // values in P.E) and run the score exchange, so that the DSMEM transfer
      // of S(i) overlaps the softmax of tile i - 1.  A tile is released two
      // tiles ahead of the exchange, which waits on the MMA.
      const int hq = ((warp & 3) * 32) + lane;
      int next_fix = 0;
      bool ok = true;
      for (int i = 0; i < n_my && ok; ++i) {
        for (; next_fix < n_my && next_fix <= i + 2; ++next_fix) {
          const int j = next_fix, s = j % kStages;
          const uint32_t tile = base + kOffE + s * kEBytes;
          const Tile tl = tile_of(t0 + j, nt_main, n_sel, n_win);
          // A full tile needs no fix-up: e_full only keeps its phase count
          // (the MMA waits for the TMA bytes itself), so the exchange below
          // never waits for memory.
          if (tl.valid < kTile) {
            if (!mbar_wait(&bars[B_TMA + s], (j / kStages) & 1, a.st, abort_p, 22)) {
              ok = false;
              break;
            }
            for (int e = p; e < (kTile - tl.valid) * 32; e += 128) {
              const int r = tl.valid + (e >> 5), cc = e & 31;
              st_shared_v4(sw128(tile + (cc >> 3) * 8192, r, cc & 7), make_uint4(0, 0, 0, 0));
            }
            fence_proxy_async_smem();
          }
          mbar_arrive(&bars[B_EFULL + s]);
          if (p == 0) progress(a.st, prog, 5);
        }
        if (!ok || !mbar_wait(&bars[B_SFULL + (i & 1)], (i >> 1) & 1, a.st, abort_p, 33)) break;
        tc_fence_after();
        send_scores(i, hq);
        tc_fence_before();
        mbar_arrive(&bars[B_XREAD + (i & 1)]);   // S(i) may now be overwritten by P(i)
        mbar_arrive_remote(mapa(smem_u32(&bars[B_XFULL + i % kXBufs]), peer));
      }
    }
    // Gathered rows.  copies(i) copies tile i's raw bytes with cp.async into
    // its stage buffer (BF16 rows straight to their swizzled place, quantised
    // rows to the staging area), up to kAhead tiles ahead; finish(i) waits
    // for them and, for quantised rows, dequantises in place: every thread
    // first reads its raw chunks, the producers meet, then BF16 is written
    // over the buffer.
    constexpr int kAhead = 3;
    constexpr int U = (kTile * (FMT == CKV_FMT_BF16 ? 32 : FMT == CKV_FMT_MIXED ? 20 : 8) + 127) / 128;
    uint32_t* vmask_s = reinterpret_cast<uint32_t*>(gbase + kOffVmask);
    int32_t* rsrc = reinterpret_cast<int32_t*>(gbase + kOffRowSrc);
    // selected entry (or row) feeding row r of tile i, before range checks
    auto raw_index = [&](int i, int r) -> int32_t {
      if (i >= n_my) return -1;
      const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
      if (r >= tl.valid) return -1;
      if (tl.win) return tl.start + r;
      return idx_b ? __ldg(idx_b + tl.start + r) : tl.start + r;
    };
    // row of the plane (dense or through the block table) feeding row r of
    // tile i from its raw index, -1 for none, published with the tile's
    // validity mask (warp-uniform i)
    auto publish = [&](int i, int r, int32_t x) {
      const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
      if (!tl.win && x >= a.kv_cap) {
        if (half == 0) report(a.st, CKV_ERR_DEVICE_BOUNDS, x);
        x = -1;
      }
      int32_t e = -1;
      if (x >= 0) {
        const int64_t row = tl.win ? (int64_t)b * a.win_cap + x
                                   : plane_row(a.kv_bt, a.kv_page, a.kv_bt_cols, a.kv_cap, b, x);
        if (!tl.win && (row < 0 || row >= a.kv_rows)) {   // a page id beyond the plane
          if (half == 0) report(a.st, CKV_ERR_DEVICE_BOUNDS, x);
        } else {
          e = (int32_t)row;
        }
      }
      rsrc[(i % kStages) * 64 + r] = e;
      const uint32_t bal = __ballot_sync(0xffffffffu, e >= 0);
      if ((r & 31) == 0) vmask_s[(i % kStages) * 2 + (r >> 5)] = bal;
    };
    // the copies of tile i (rows published, stage free).  BF16 rows go by
    // TMA gathers of four rows each, issued by one thread per warp, straight
    // to their swizzled place.  Quantised rows and their scales go by
    // cp.async into the staging area, 16 bytes (MIXED scale words: 4 bytes,
    // a row stride TMA cannot address) a copy, every producer thread
    // issuing its own chunks: they need no tensor map and complete under the
    // thread's cp.async groups, which finish(i) waits for.
    auto copies = [&](int i) {
      const int s = i % kStages;
      if (p == 0 && i < 4) trace(a.st, tr, 49 + i, tr0);
      const uint32_t tile = base + kOffE + s * kEBytes;
      const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
      const int32_t* rs = rsrc + s * 64;
      if constexpr (FMT == CKV_FMT_BF16) {
        const CUtensorMap* gm = &a.gmap[tl.win ? 2 : 0];
        if ((p & 31) == 0) {
          // lane 0 of each producer warp issues four of the sixteen groups;
          // warp 0's also arms the barrier (the transaction count may go
          // negative until it does)
          if (p == 0) mbar_expect_tx(&bars[B_GFULL + s], 64u * 512u);
#pragma unroll 1
          for (int g = (p >> 5) * 4; g < (p >> 5) * 4 + 4; ++g) {
            int y[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // an empty row reads the plane's first row (a valid address)
              // and is zeroed from the mask
              const int32_t e = rs[4 * g + k];
              y[k] = e >= 0 ? e : 0;
            }
#pragma unroll
            for (int kc = 0; kc < 4; ++kc)
              tma_gather4(tile + kc * 8192 + g * 512, gm, half * 256 + kc * 64, y[0], y[1], y[2], y[3],
                          &bars[B_GFULL + s]);
          }
        }
      } else {
        const uint8_t* data = tl.win ? a.win_data : a.kv_data;
        constexpr int kRowBytes = FMT == CKV_FMT_MIXED ? 576 : 256;
        const int hoff = FMT == CKV_FMT_MIXED ? half * 256 : half * 128;
        const int hbytes = FMT == CKV_FMT_MIXED ? (half == 0 ? 256 : 320) : 128;
        const uint32_t raw0 = tile + (FMT == CKV_FMT_MIXED ? kRawOffMixed : kRawOffFp4);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = p + 128 * u;
          if (j < kTile * J) {
            const int r = chunk_row<FMT>(j, half), q = j - r * J;
            const int32_t e = rs[r];
            if (e >= 0) cp_async16(raw0 + r * hbytes + q * 16, data + (int64_t)e * kRowBytes + hoff + q * 16);
          }
        }
        const uint8_t* scale = static_cast<const uint8_t*>(tl.win ? a.win_scale : a.kv_scale);
        if constexpr (FMT == CKV_FMT_MIXED) {
          // row p's scale words for this half (at most 4: nope_block is 448 or 64)
          if (p < 64 && rs[p] >= 0) {
            const int64_t ent = rs[p];
            const int nblk = 448 / a.nope_block, nb0 = (half * 256) / a.nope_block;
            const int nb1 = (half * 256 + (half == 0 ? 256 : 192) - 1) / a.nope_block;
            for (int k = 0; k <= nb1 - nb0; ++k)
              cp_async4(tile + kScaleOffMixed + p * 32 + k * 4, scale + (ent * nblk + nb0 + k) * 4);
          }
        } else {
          // row p's 16 scale bytes of this half, in 128-byte groups of four rows
          if (p < 64 && rs[p] >= 0)
            cp_async16(tile + kScaleOffFp4 + (p >> 2) * 128 + (p & 3) * 16, scale + (int64_t)rs[p] * 32 + half * 16);
        }
      }
      cp_async_commit();
    };
    auto finish = [&](int i, int newer) -> bool {
      const int s = i % kStages;
      const uint32_t tile = base + kOffE + s * kEBytes;
      bool landed = FMT != CKV_FMT_BF16 || mbar_wait(&bars[B_GFULL + s], (i / kStages) & 1, a.st, abort_p, 35);
      cp_async_wait(newer);                      // this thread's copies of tile i
      if (!bar_and(2, 128, landed)) return false;   // everyone's
      if (p == 0 && i < 2) trace(a.st, tr, 51 + i, tr0);   // debug: data landed
      const bool nb64 = a.nope_block == 64;
      if constexpr (FMT == CKV_FMT_BF16) {
        // empty rows: zero their bytes so that P = 0 meets finite values
        const uint64_t vbits = (uint64_t)vmask_s[s * 2] | ((uint64_t)vmask_s[s * 2 + 1] << 32);
        if (vbits != ~0ull) {
          for (int e = p; e < kTile * 32; e += 128) {
            const int r = e >> 5, cc = e & 31;
            if (!((vbits >> r) & 1ull))
              st_shared_v4(sw128(tile + (cc >> 3) * 8192, r, cc & 7), make_uint4(0, 0, 0, 0));
          }
        }
      } else {
        const uint64_t vbits = (uint64_t)vmask_s[s * 2] | ((uint64_t)vmask_s[s * 2 + 1] << 32);
        Raw raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = p + 128 * u;
          raw[u].v = make_uint4(0u, 0u, 0u, 0u);
          raw[u].s = 0u;
          if (j < kTile * J) {
            const int r = chunk_row<FMT>(j, half), q = j - r * J;
            if ((vbits >> r) & 1ull) {
              if constexpr (FMT == CKV_FMT_MIXED) {
                raw[u].v = ld_shared_u4(tile + kRawOffMixed + r * (half == 0 ? 256 : 320) + q * 16);
                if (q < (half == 0 ? 16 : 12)) {
                  // nope_block is 448 (one scale word) or 64: no division
                  const int blk = nb64 ? ((half * 256 + q * 16) >> 6) - ((half * 256) >> 6) : 0;
                  raw[u].s = ld_shared_u32(tile + kScaleOffMixed + r * 32 + blk * 4);
                }
              } else {
                raw[u].v = ld_shared_u4(tile + kRawOffFp4 + r * 128 + q * 16);
                raw[u].s = ld_shared_u16(tile + kScaleOffFp4 + (r >> 2) * 128 + (r & 3) * 16 + q * 2);
              }
            }
          }
        }
        asm volatile("bar.sync 2, 128;" ::: "memory");   // raw bytes read: overwrite
        if (p == 0 && i < 2) trace(a.st, tr, 55 + i, tr0);   // debug: raw read
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = p + 128 * u;
          if (j < kTile * J) {
            const int r = chunk_row<FMT>(j, half), q = j - r * J;
            store_chunk<FMT>(a, tile, r, q, raw[u], half);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[B_EFULL + s]);
      if (p == 0) progress(a.st, prog, 5);
      if (p == 0 && i < 4) trace(a.st, tr, 53 + i, tr0);
      return true;
    };
    if (!use_tma) {
      // the first kAhead + 1 tiles (free stages): every lookup in one round
      // trip (thread p takes row p % 64 of tiles p / 64 and p / 64 + 2)
      const int n_init = min(n_my, kAhead + 1);
      {
        const int r = p & 63, ta = p >> 6, tb = ta + 2;
        const int32_t xa = ta < n_init ? raw_index(ta, r) : -1;
        const int32_t xb = tb < n_init ? raw_index(tb, r) : -1;
        if (ta < n_init) publish(ta, r, xa);
        if (tb < n_init) publish(tb, r, xb);
      }
      int32_t x_next = p < 64 ? raw_index(n_init, p) : -1;   // used one tile later
      asm volatile("bar.sync 2, 128;" ::: "memory");
      if (p == 0) trace(a.st, tr, 3, tr0);   // debug: first rows published
      for (int t = 0; t < n_init; ++t) copies(t);
      if (p == 0) trace(a.st, tr, 7, tr0);   // debug: first copies issued
      int issued = n_init, finished = 0;
      bool ok = true;
      for (int i = 0; i < n_my && ok; ++i) {
        ok = finish(i, issued - 1 - i);
        if (!ok) break;
        finished = i + 1;
        if (issued < n_my) {
          const int t = issued, s = t % kStages;
          ok = t < kStages ||
               mbar_wait(&bars[B_EEMPTY + s], ((t / kStages) + 1) & 1, a.st, abort_p, 23);
          ok = bar_and(2, 128, ok);   // every producer leaves together on a failed wait
          if (!ok) break;
          if (p < 64) {
            publish(t, p, x_next);
            x_next = raw_index(t + 1, p);
          }
          asm volatile("bar.sync 2, 128;" ::: "memory");
          copies(t);
          ++issued;
        }
      }
      cp_async_wait(0);   // nothing stays in flight past this point
      if (FMT == CKV_FMT_BF16 && p == 0 && finished < issued) {
        // a wait failed: let the gathers already issued land (bounded)
        // before this CTA can exit
        volatile int keep_waiting = 0;
        for (int t = finished; t < issued; ++t)
          mbar_wait(&bars[B_GFULL + t % kStages], (t / kStages) & 1, a.st, &keep_waiting, 36);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      const uint32_t tO = tmem + kColO, tQ = tmem + kColQ;
      auto issue_pv = [&](int j) -> bool {
        const int sj = j % kStages, bj = j & 1;
        if (!mbar_wait(&bars[B_PFULL + bj], (j >> 1) & 1, a.st, abort_p, 24)) return false;
        tc_fence_after();
        if ((unsigned)(j - toff) < 8u) trace(a.st, tr, 17 + j - toff, tr0);
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
        if (use_tma && !mbar_wait(&bars[B_TMA + s], (i / kStages) & 1, a.st, abort_p, 37)) break;
        tc_fence_after();
        if (use_tma && (unsigned)(i - toff) < 8u) trace(a.st, tr, 49 + i - toff, tr0);   // the tile's bytes have landed
        if ((unsigned)(i - toff) < 8u) trace(a.st, tr, 1 + i - toff, tr0);
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint32_t kc = ks >> 2, w = ks & 3;
          const uint64_t db = smem_desc(tile + kc * 8192 + w * 32, 16, 1024, 2);
          umma_f16_ta(tmem + kColS + 64 * bi, tQ + 8 * ks, db, kIdescQK, ks > 0);
        }
        umma_commit(&bars[B_SFULL + bi]);
        progress(a.st, prog, 1);
        if ((unsigned)(i - toff) < 8u) trace(a.st, tr, 9 + i - toff, tr0);
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
    // Partial scores of tile i: the exchange warps send S(i) for TMA-fed
    // tiles; for gathered tiles this thread sends its own row first.
    bool ok = true;
    for (int i = 0; i < n_my && ok; ++i) {
      const int bi = i & 1;
      const uint32_t tS = tmem + kColS + 64 * bi + lane_base;
      if (!mbar_wait(&bars[B_SFULL + bi], (i >> 1) & 1, a.st, abort_p, 26)) break;
      tc_fence_after();
      if (h == 0) progress(a.st, prog, 2);
      if (h == 0 && (unsigned)(i - toff) < 8u) trace(a.st, tr, 25 + i - toff, tr0);
      if (!use_tma) {
        send_scores(i, h);
        mbar_arrive_remote(mapa(smem_u32(&bars[B_XFULL + i % kXBufs]), peer));
        if (h == 0 && i < 2) trace(a.st, tr, 5 + i, tr0);   // debug: S(i) sent
      }
      const Tile tl = tile_of(t0 + i, nt_main, n_sel, n_win);
      // validity of the tile's rows (selected entries may be -1 / out of range)
      uint64_t vmask = tl.valid >= 64 ? ~0ull : ((1ull << tl.valid) - 1ull);
      if (!use_tma) {
        // the producers' mask of tile i (their e_full arrive released it)
        const int s = i % kStages;
        mbar_wait(&bars[B_EFULL + s], (i / kStages) & 1, a.st, abort_p, 32);
        const uint32_t* vm = reinterpret_cast<const uint32_t*>(gbase + kOffVmask) + s * 2;
        vmask = (uint64_t)vm[0] | ((uint64_t)vm[1] << 32);
      }
      const uint32_t xi = i % kXBufs;
      if (!mbar_wait_poll(&bars[B_XFULL + xi], (i / kXBufs) & 1, a.st, abort_p, 27)) break;
      if (h == 0) progress(a.st, prog, 3);
      if (h == 0 && (unsigned)(i - toff) < 8u) trace(a.st, tr, 33 + i - toff, tr0);
      const uint32_t xrow = base + kOffX + xi * kXBytes + h * 128;
      // Raw scores of row h: s_j = own_j + peer_j (own: S(i) in TMEM, fp32;
      // peer: its fp16 partial), -inf for an invalid column.  All 64 stay in
      // registers; z_j = s_j * scale * log2(e) is folded into the exponent.
      float sv[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tS, r0);
        tmem_ld32(tS + 32, r1);
        float4 o[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) o[c] = ld_shared_v4f(xrow + ((c ^ (h & 7)) << 4));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float ow[4] = {o[c].x, o[c].y, o[c].z, o[c].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 8 * c + 2 * u;
            const uint32_t pwd = __float_as_uint(ow[u]);
            const float2 pf = __half22float2(*reinterpret_cast<const __half2*>(&pwd));
            const uint32_t o0 = j < 32 ? r0[j] : r1[j - 32], o1 = j < 32 ? r0[j + 1] : r1[j - 31];
            sv[j] = __uint_as_float(o0) + pf.x;
            sv[j + 1] = __uint_as_float(o1) + pf.y;
          }
        }
      }
      if (vmask != ~0ull) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!((vmask >> j) & 1ull)) sv[j] = -INFINITY;
      }
      float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
      for (int j = 4; j < 64; ++j) mx[j & 3] = fmaxf(mx[j & 3], sv[j]);
      // scale_log2 > 0 (checked on the host), so max z = max s * scale_log2
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
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
      // the exchange warps must have read S(i) before P(i) overwrites it
      if (use_tma && !mbar_wait(&bars[B_XREAD + bi], (i >> 1) & 1, a.st, abort_p, 34)) break;
      // P(i) = 2^(z - m) as bf16 pairs over columns 0 .. 31 of this S
      // buffer; l sums the unrounded p
      uint32_t pk[32];
      if (m_used == -INFINITY) {
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = 0u;
      } else {
        const float negm = -m_used;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float p0 = fast_exp2(fmaf(sv[2 * k], a.scale_log2, negm));
          const float p1 = fast_exp2(fmaf(sv[2 * k + 1], a.scale_log2, negm));
          ls[k & 3] += p0 + p1;
          __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          pk[k] = *reinterpret_cast<uint32_t*>(&pb);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      }
      tmem_st32(tS, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[B_PFULL + bi]);
      if (h == 0) progress(a.st, prog, 8);
      if (h == 0 && (unsigned)(i - toff) < 8u) trace(a.st, tr, 41 + i - toff, tr0);
    }
    if (n_my > 0) {
      // s_full of the last tile implies every PV up to n_my - 3 is done, so
      // o_done may still owe two phases: wait for them in order (a single
      // parity wait could alias the older one).
      if (n_my >= 2) mbar_wait(&bars[B_ODONE], (n_my - 2) & 1, a.st, abort_p, 29);
      mbar_wait(&bars[B_ODONE], (n_my - 1) & 1, a.st, abort_p, 29);
      tc_fence_after();
    }
    // this CTA's partial -> workspace: O / l rounded to fp16 (bounded by the
    // largest |e|, so fp16's range holds it) and (m, l) in f32, laid out
    // [8-column chunk][head] so that every store and load is coalesced
    uint4* po = reinterpret_cast<uint4*>(a.part) +
                (((int64_t)blockIdx.z * gridDim.y + b) * (2 * G) + blockIdx.x) * (kPartFloats / 4);
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    uint4* pw = po + h;
#pragma unroll 1
    for (int c = 0; c < 8; ++c, pw += 4 * 128) {
      uint32_t r[32];
      if (n_my > 0) {
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __half2 hv = __floats2half2_rn(__uint_as_float(r[8 * k + 2 * e]) * inv_l,
                                         __uint_as_float(r[8 * k + 2 * e + 1]) * inv_l);
          w[e] = *reinterpret_cast<uint32_t*>(&hv);
        }
        __stcg(pw + k * 128, make_uint4(w[0], w[1], w[2], w[3]));
      }
    }
    reinterpret_cast<float2*>(po + 32 * 128)[h] = make_float2(m_used, l);
    // No fence here: the CTA barrier below orders these stores before the
    // cluster barrier's release (a sequence-wide cluster) or before thread
    // 0's fence and counter increment (pair clusters).
    if (h == 0 && !use_tma) trace(a.st, tr, 11, tr0);   // debug: partial stored
  }
  tc_fence_before();
  if (tid == 0) progress(a.st, prog, 6);
  if (tid == 8 * 32) trace(a.st, tr, 57, tr0);   // a softmax thread (h = 64)
  if (tid == 8 * 32) stamp3(1);
  // The cluster meets once more: no CTA exits while another may still touch
  // its shared memory, and with a sequence-wide cluster every partial of the
  // sequence is written once it is through.
  cluster_barrier(&bars[B_CLUSTER], a.cluster_all ? 2 * a.G : 2, a.st, abort_p, 30);
  if (tid == 0) trace(a.st, tr, 58, tr0);
  pdl_launch_dependents();

  // ------------------------------------ merge of the G partials of half c ----
  // With a sequence-wide cluster every partial of the sequence is written
  // once the cluster barrier above is through, and pair `pair` merges units
  // [u0, u1) of 8 columns of its half (merge_partials).
  // With pair clusters, no CTA waits for another cluster: each CTA counts
  // itself in on its half's counter once its partial is written, and the
  // last of the G CTAs of a half merges all 32 units of that half (and
  // resets the counter for the next call).  A launch therefore never depends
  // on CTAs outside its own clusters being resident.
  uint32_t* cnt = a.tickets + ((int64_t)blockIdx.z * gridDim.y + b) * 2;
  __shared__ int merge_here;
  if (tid == 0) {
    int last = 1;
    if (!a.cluster_all) {
      __threadfence();   // this CTA's partial (ordered before by the CTA barrier) before its count
      last = atomicAdd(cnt + half, 1u) == (uint32_t)(G - 1);
      if (last) {
        __threadfence();   // the other CTAs' partials, released by their counts, after ours
        cnt[half] = 0u;
      }
    }
    merge_here = last;
  }
  __syncthreads();
  if (tid == 0) stamp3(2);
  if (tid == 0 && !use_tma) trace(a.st, tr, 13, tr0);   // debug: every partial of the half written
  if (!*abort_p && merge_here) {
    const uint4* pq0 = reinterpret_cast<const uint4*>(a.part) +
                       (((int64_t)blockIdx.z * gridDim.y + b) * (2 * G) + half) * (kPartFloats / 4);
    // the tile ring is dead by now: weights, then the staged pieces
    float* wsm = reinterpret_cast<float*>(gbase + kOffE);
    const uint32_t stage = base + kOffE + kMergeWBytes;
    // one CTA of half 0 writes the lse
    const bool lse_here = a.cluster_all ? blockIdx.x == 0 : half == 0;
    float* lse = lse_here && a.lse ? a.lse + (int64_t)b * a.H : nullptr;
    __nv_bfloat16* out = a.out + (int64_t)b * a.H * 512 + half * 256;
    const int u0 = a.cluster_all ? pair * 32 / G : 0, u1 = a.cluster_all ? (pair + 1) * 32 / G : 32;
    const float2* rtab = (half == 1 && a.rope_pos && a.rope_out)
                             ? reinterpret_cast<const float2*>(gbase + kOffRope) : nullptr;
    merge_partials(pq0, wsm, stage, G, a.H, out, lse, tid, u0, u1, rtab);
    if (tid == 0 && !use_tma) trace(a.st, tr, 4, tr0);   // debug: merge done
  }
  __syncthreads();
  if (tid == 0) stamp3(3);

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0) progress(a.st, prog, 7);
  if (tid == 0) trace(a.st, tr, 59, tr0);
  if (tr && tid == 0) a.st->pad[60] = n_my;
}

namespace {

// 2-D map over a BF16 plane viewed as [rows][512] bf16, box 64 x 64, 128B swizzle.
bool encode_bf16_rows(CUtensorMap* m, const void* data, int64_t rows) {
  if (rows <= 0 || rows >= ((int64_t)1 << 31)) return false;
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, data, 512, (uint64_t)rows, 1024, 64, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

// 2-D map of one-row boxes over a plane's rows (`rows` rows of `row_elems`
// elements of `dt`, contiguous) for TMA gathers of `box_elems` elements.
bool encode_gather_rows(CUtensorMap* m, const void* data, CUtensorMapDataType dt, int elem_bytes,
                        int64_t rows, int row_elems, int box_elems, CUtensorMapSwizzle sw) {
  if (!data || rows <= 0 || rows >= ((int64_t)1 << 31)) return false;
  return encode_tmap_2d(m, dt, data, (uint64_t)row_elems, (uint64_t)rows,
                        (uint64_t)row_elems * elem_bytes, (uint32_t)box_elems, 1, sw);
}

// The gather maps of one layer: [0, 1] main plane, [2, 3] window plane.
// BF16: 64-element boxes, 128-byte swizzle (straight into the MMA tile);
// MIXED: 256- and 320-byte boxes (the two halves' bytes, as 16-bit
// elements); FP4: 128-byte code boxes and 16-byte scale boxes.
bool encode_gather_maps(AttnArgs& a, int B) {
  const uint8_t* data[2] = {a.kv_data, a.win_data};
  const int64_t rows[2] = {a.kv_rows, (int64_t)B * a.win_cap};
  for (int k = 0; k < 2; ++k) {
    CUtensorMap* m = &a.gmap[2 * k];
    if (!encode_gather_rows(m, data[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows[k], 512, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    m[1] = m[0];
  }
  return true;
}

}  // namespace

using AttnKernelFn = void (*)(const CUtensorMap, const CUtensorMap, const AttnBatch);

// The kernel instance for a cache format (nullptr for an unknown one), with
// its launch attributes set once per device.
static AttnKernelFn attn_kernel_for(int fmt) {
  static DeviceOnce once;
  const AttnKernelFn ks[3] = {attn_kernel<CKV_FMT_BF16>, attn_kernel<CKV_FMT_MIXED>,
                              attn_kernel<CKV_FMT_FP4>};
  const cudaError_t e = once_per_device(once, [&](int) {
    for (AttnKernelFn k : ks) {
      cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAttn);
      if (r == cudaSuccess) r = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return nullptr;
  return fmt == CKV_FMT_BF16 ? ks[0] : fmt == CKV_FMT_MIXED ? ks[1] : fmt == CKV_FMT_FP4 ? ks[2] : nullptr;
}

cudaError_t launch_attention_layers(const AttnArgs* layers, int n, int B, cudaStream_t stream) {
  if (n < 1 || n > kLayersPerLaunch) return cudaErrorInvalidValue;
  const AttnArgs& a0 = layers[0];
  for (int l = 1; l < n; ++l)
    if (layers[l].fmt != a0.fmt || layers[l].G != a0.G || layers[l].cluster_all != a0.cluster_all)
      return cudaErrorInvalidValue;
  const AttnKernelFn kern = attn_kernel_for(a0.fmt);
  if (!kern) return cudaErrorInvalidValue;
  AttnBatch batch;
  memset(&batch, 0, sizeof(batch));
  for (int l = 0; l < n; ++l) {
    batch.layer[l] = layers[l];
    batch.layer[l].use_tma = 0;
    batch.layer[l].tag = kArgsTag ^ l;
  }
  CUtensorMap mk, mw;
  memset(&mk, 0, sizeof(mk));
  memset(&mw, 0, sizeof(mw));
  // Contiguous BF16 rows (HCA, one layer) stream through TMA; gathered or
  // quantised rows go through the producer warps.
  if (n == 1 && a0.fmt == CKV_FMT_BF16 && a0.idx == nullptr &&
      encode_bf16_rows(&mk, a0.kv_data, a0.kv_rows) &&
      encode_bf16_rows(&mw, a0.win_data, (int64_t)B * a0.win_cap))
    batch.layer[0].use_tma = 1;
  // BF16 layers gather their rows with TMA (quantised rows go by cp.async)
  for (int l = 0; l < n; ++l)
    if (!batch.layer[l].use_tma && batch.layer[l].fmt == CKV_FMT_BF16 &&
        !encode_gather_maps(batch.layer[l], B))
      return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a0.G, B, n);
  cfg.blockDim = dim3(kThreadsAttn, 1, 1);
  cfg.dynamicSmemBytes = kSmemAttn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a0.cluster_all ? 2 * a0.G : 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, mk, mw, batch);
}

// Clusters of `cluster_size` CTAs of attn_kernel that fit on the GPU at once
// (cached per device and size).
int attn_max_active_clusters(int cluster_size) {
  // every cluster size 1 .. 2 kMaxPairs, asked once per device
  static DeviceOnce once;
  static int cache[kOnceDevices][2 * kMaxPairs + 1];
  if (cluster_size < 1 || cluster_size > 2 * kMaxPairs) return 0;
  int dev = -1;
  const cudaError_t e = once_per_device(once, [&](int d) {
    dev = d;
    // every format's instance has the same resources: ask about one
    const AttnKernelFn kern = attn_kernel_for(CKV_FMT_MIXED);
    for (int cs = 0; cs <= 2 * kMaxPairs; ++cs) {
      int n = 0;
      if (kern && cs >= 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs, 1, 1);
        cfg.blockDim = dim3(kThreadsAttn, 1, 1);
        cfg.dynamicSmemBytes = kSmemAttn;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
          (void)cudaGetLastError();
          n = 0;
        }
      }
      cache[d][cs] = n;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return 0;
  if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) return 0;
  return cache[dev][cluster_size];
}

cudaError_t launch_attention(const AttnArgs& a, int B, cudaStream_t stream) {
  return launch_attention_layers(&a, 1, B, stream);
}

}  // namespace ckv

// csa_sparse_attn / hca_attn: shared-KV decode attention on tcgen05.
//
// "DeepSeek-V4 KV Cache 深度分析": §五 -- each compressed entry is both key
// and value (o = sum_j a_j C_j); §十一 -- Attention(Q, selected) followed by
// the 128-token window; §三 -- HCA attends densely to every ratio-128 entry
// plus the window.  One softmax over the union of the rows (no sink).
//
// Decomposition (per sequence b, one thread-block cluster of 2G CTAs):
//   * CTA (pair p, half c) owns latent dims [256c, 256c + 256).  Its
//     accumulator O_c = 128 heads x 256 f32 lives in TMEM columns [0, 256);
//     a 128 x 64 f32 score tile S lives in columns [256, 320).
//   * Pair p walks a contiguous range of 64-row tiles of the row list
//     (selected entries, then window slots).  For each tile both CTAs compute
//     the partial product S_c = Q[:, half c] . E[:, half c]^T (tcgen05,
//     K = 256), swap S_c over distributed shared memory and add, so both hold
//     the same S = S_0 + S_1 bit for bit and run the same online softmax;
//     then each accumulates O_c += P . E[:, half c] (tcgen05, N = 256).
//   * At the end the G pairs merge their (m, l, O) in the cluster: CTA
//     (p, c) finalises latent columns [256c + p*256/G, ...) from the G
//     partial accumulators of half c read over DSMEM, and writes bf16 o.
// Rows are dequantised (FP8 x scale / FP4 x scale / BF16) into bf16 shared
// memory tiles laid out in the 128-byte-swizzled K-major form the tensor core
// reads; the same tile serves as the K-major B operand of Q.E^T and the
// MN-major B operand of P.E.

#include "common.cuh"
#include "attention.cuh"

namespace ckv {

namespace {

constexpr int kTile = 64;           // rows per tile
constexpr int kStages = 2;          // E tile pipeline depth
constexpr int kThreadsAttn = 288;   // 4 softmax warps, 4 producer warps, 1 MMA warp
constexpr uint32_t kQBytes = 128 * 256 * 2;           // 64 KB
constexpr uint32_t kEBytes = kTile * 256 * 2;         // 32 KB
constexpr uint32_t kPBytes = 128 * kTile * 2;         // 16 KB
constexpr uint32_t kXBytes = 128 * kTile * 4;         // 32 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffE = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffE + kStages * kEBytes;
constexpr uint32_t kOffX = kOffP + kPBytes;
constexpr uint32_t kOffO = kOffE;                     // final O staging reuses E/P/X
constexpr uint32_t kOffML = kOffX + 2 * kXBytes;      // m, l per head
constexpr uint32_t kOffRows = kOffML + 128 * 8;       // selected entry per row
constexpr uint32_t kOffBar = kOffRows + kMaxTopk * 4;
constexpr uint32_t kNumBars = 10;
constexpr uint32_t kOffSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffSlot + 16;
constexpr uint32_t kSmemAttn = kSmemUsed + 1024;      // alignment slack
static_assert(kOffE + 128 * 256 * 4 <= kOffML, "O staging fits in the E/P/X region");
static_assert(kSmemAttn <= 232448, "fits the 227 KB opt-in limit");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;
constexpr uint32_t kIdescQK = idesc_bf16(128, kTile, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, 0, 1);

enum { B_EFULL0 = 0, B_EFULL1, B_EEMPTY0, B_EEMPTY1, B_SFULL, B_PFULL, B_ODONE, B_XFULL0, B_XFULL1 };

struct RowSrc {
  const uint8_t* data;
  const void* scale;
  int64_t entry;  // global slot (b * cap + pos), or -1 when the row is empty
};

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

// Dequantise local latent chunk `q` of row `src` (half `half`) into the bf16
// tile `tile` at row `r`.  Writes zeros for an empty row.
__device__ __forceinline__ void fill_chunk(const AttnArgs& a, uint32_t tile, int r, int q,
                                           const RowSrc& src, int half) {
  const bool empty = src.entry < 0;
  if (a.fmt == CKV_FMT_BF16) {
    // 32 chunks of 8 bf16
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

__global__ void __launch_bounds__(kThreadsAttn, 1) attn_kernel(AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(gbase + kOffSlot);
  int32_t* rows = reinterpret_cast<int32_t*>(gbase + kOffRows);
  float2* ml = reinterpret_cast<float2*>(gbase + kOffML);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)(rank >> 1), half = (int)(rank & 1);
  const uint32_t peer = rank ^ 1u;
  const int b = blockIdx.y;
  const int G = a.G;

  // Row list of this sequence: n_sel selected entries, then n_win window slots.
  const int n_sel = a.idx ? a.topk : max(0, min(a.n_comp[b], a.n_comp_max));
  const int n_win = max(0, min(a.win_len[b], (int)a.win_cap));
  const int n_rows = n_sel + n_win;
  const int n_tiles = (n_rows + kTile - 1) / kTile;
  const int t0 = (int)((int64_t)pair * n_tiles / G), t1 = (int)((int64_t)(pair + 1) * n_tiles / G);
  const int n_my = t1 - t0;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bars[B_EFULL0], 128);
    mbar_init(&bars[B_EFULL1], 128);
    mbar_init(&bars[B_EEMPTY0], 1);
    mbar_init(&bars[B_EEMPTY1], 1);
    mbar_init(&bars[B_SFULL], 1);
    mbar_init(&bars[B_PFULL], 128);
    mbar_init(&bars[B_ODONE], 1);
    mbar_init(&bars[B_XFULL0], 128);
    mbar_init(&bars[B_XFULL1], 128);
    fence_mbar_init();
  }
  if (warp == 8) tmem_alloc(tslot, kTmemCols);
  if (warp >= 4 && warp < 8) {
    const int p = tid - 128;
    // Q[b, :, half] -> swizzled K-major tiles (rows >= H are zero)
    for (int j = p; j < 128 * 32; j += 128) {
      const int h = j >> 5, cc = j & 31;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (h < a.H)
        v = *reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.H + h) * 512 + half * 256 + cc * 8);
      st_shared_v4(sw128(base + kOffQ + (cc >> 3) * 16384, h, cc & 7), v);
    }
    if (a.idx) {
      for (int j = p; j < a.topk; j += 128) {
        int e = a.idx[(int64_t)b * a.topk + j];
        if (e >= a.kv_cap) {
          report(a.st, CKV_ERR_DEVICE_BOUNDS, e);
          e = -1;
        }
        rows[j] = e;
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  volatile int* abort_p = &abort_flag;

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------ producers ----
    const int p = tid - 128;
    const int J = chunks_per_row(a.fmt, half);
    for (int i = 0; i < n_my; ++i) {
      const int s = i & 1;
      if (i >= kStages && !mbar_wait(&bars[B_EEMPTY0 + s], ((i >> 1) + 1) & 1, a.st, abort_p, 1)) break;
      const uint32_t tile = base + kOffE + s * kEBytes;
      const int r0 = (t0 + i) * kTile;
      for (int j = p; j < kTile * J; j += 128) {
        const int r = j / J, q = j - r * J;
        const int row = r0 + r;
        RowSrc src;
        src.entry = -1;
        if (row < n_sel) {
          const int64_t e = a.idx ? rows[row] : row;
          if (e >= 0) {
            src.data = a.kv_data;
            src.scale = a.kv_scale;
            src.entry = (int64_t)b * a.kv_cap + e;
          }
        } else if (row < n_rows) {
          src.data = a.win_data;
          src.scale = a.win_scale;
          src.entry = (int64_t)b * a.win_cap + (row - n_sel);
        }
        fill_chunk(a, tile, r, q, src, half);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[B_EFULL0 + s]);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      const uint32_t tS = tmem + kColS, tO = tmem + kColO;
      for (int i = 0; i < n_my; ++i) {
        const int s = i & 1;
        const uint32_t tile = base + kOffE + s * kEBytes;
        if (!mbar_wait(&bars[B_EFULL0 + s], (i >> 1) & 1, a.st, abort_p, 2)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint32_t kc = ks >> 2, w = ks & 3;
          const uint64_t da = smem_desc(base + kOffQ + kc * 16384 + w * 32, 16, 1024, 2);
          const uint64_t db = smem_desc(tile + kc * 8192 + w * 32, 16, 1024, 2);
          umma_f16(tS, da, db, kIdescQK, ks > 0);
        }
        umma_commit(&bars[B_SFULL]);
        if (!mbar_wait(&bars[B_PFULL], i & 1, a.st, abort_p, 3)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t da = smem_desc(base + kOffP + ks * 32, 16, 1024, 2);
          const uint64_t db = smem_desc(tile + ks * 2048, 8192, 1024, 2);
          umma_f16(tO, da, db, kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_ODONE]);
        umma_commit(&bars[B_EEMPTY0 + s]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax (row = head) ----
    const int h = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + kColS + lane_base, tO = tmem + kColO + lane_base;
    float m = -INFINITY, l = 0.f;
    for (int i = 0; i < n_my; ++i) {
      if (!mbar_wait(&bars[B_SFULL], i & 1, a.st, abort_p, 4)) break;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld();
      // swap the partial scores with the other half of the pair
      const int x = i & 1;
      const uint32_t xrow = base + kOffX + x * kXBytes + h * 256;
      const uint32_t xrow_peer = mapa(xrow, peer);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_cluster_v4(xrow_peer + ((c ^ (h & 7)) << 4),
                      make_float4(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1]),
                                  __uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3])));
      mbar_arrive_remote(mapa(smem_u32(&bars[B_XFULL0 + x]), peer));
      if (!mbar_wait(&bars[B_XFULL0 + x], (i >> 1) & 1, a.st, abort_p, 5)) break;
      float z[64];
      const int r0 = (t0 + i) * kTile;
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float4 o = ld_shared_v4f(xrow + ((c ^ (h & 7)) << 4));
        const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = 4 * c + k, row = r0 + j;
          bool valid = row < n_rows;
          if (valid && row < n_sel && a.idx) valid = rows[row] >= 0;
          const float sv = __uint_as_float(sr[j]) + ov[k];
          z[j] = valid ? sv * a.scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, z[j]);
        }
      }
      const float m_new = fmaxf(m, tmax);
      if (i > 0) {
        if (!mbar_wait(&bars[B_ODONE], (i - 1) & 1, a.st, abort_p, 6)) break;
        tc_fence_after();
      }
      if (i > 0 && m_new > m && m != -INFINITY) {
        const float alpha = exp2f(m - m_new);
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
      m = m_new;
      const uint32_t prow = base + kOffP;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float p0 = m == -INFINITY ? 0.f : exp2f(z[8 * c + 2 * k] - m);
          const float p1 = m == -INFINITY ? 0.f : exp2f(z[8 * c + 2 * k + 1] - m);
          __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          const float2 pr = __bfloat1622float2(pb);
          l += pr.x + pr.y;
          pk[k] = *reinterpret_cast<uint32_t*>(&pb);
        }
        st_shared_v4(sw128(prow, h, c), make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[B_PFULL]);
    }
    if (n_my > 0) {
      mbar_wait(&bars[B_ODONE], (n_my - 1) & 1, a.st, abort_p, 7);
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
        const int c4 = c * 8 + k;  // float4 chunk 0..63 of the 256-wide row
        st_shared_v4(orow + (((c4 & ~7) | ((c4 & 7) ^ (h & 7))) << 4),
                     make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]));
      }
    }
    ml[h] = make_float2(m, l);
    tc_fence_before();
  }

  cluster_sync();

  if (warp < 4) {
    // --------------------------------------------- in-cluster merge ----
    const int h = tid;
    float mq[4], wq[4];
    float M = -INFINITY;
    for (int q = 0; q < G; ++q) {
      const uint32_t rq = 2u * q + half;
      const float2 v = make_float2(ld_cluster_f32(mapa(smem_u32(&ml[h].x), rq)),
                                   ld_cluster_f32(mapa(smem_u32(&ml[h].y), rq)));
      mq[q] = v.x;
      wq[q] = v.y;
      M = fmaxf(M, v.x);
    }
    float L = 0.f;
    for (int q = 0; q < G; ++q) {
      const float f = mq[q] == -INFINITY ? 0.f : exp2f(mq[q] - M);
      L += wq[q] * f;
      mq[q] = f;  // now the weight of partial q
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int cols = 256 / G, c4_0 = pair * cols / 4;
    if (h < a.H) {
      __nv_bfloat16* out = a.out + ((int64_t)b * a.H + h) * 512 + half * 256;
      const uint32_t orow = base + kOffO + h * 1024;
      for (int c4 = c4_0; c4 < c4_0 + cols / 4; c4 += 2) {
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int q = 0; q < G; ++q) {
          if (mq[q] == 0.f) continue;
          const uint32_t rq = 2u * q + half;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int cc = c4 + u;
            const uint32_t addr = orow + (((cc & ~7) | ((cc & 7) ^ (h & 7))) << 4);
            const float4 v = ld_cluster_v4(mapa(addr, rq));
            acc[4 * u] += mq[q] * v.x;
            acc[4 * u + 1] += mq[q] * v.y;
            acc[4 * u + 2] += mq[q] * v.z;
            acc[4 * u + 3] += mq[q] * v.w;
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
  cluster_sync();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t launch_attention(const AttnArgs& a, int B, cudaStream_t stream) {
  static int attr_done = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_done != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemAttn);
    if (e != cudaSuccess) return e;
    attr_done = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.G, B, 1);
  cfg.blockDim = dim3(kThreadsAttn, 1, 1);
  cfg.dynamicSmemBytes = kSmemAttn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * a.G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_kernel, a);
}

}  // namespace ckv

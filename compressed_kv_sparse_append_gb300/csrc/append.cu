// kv_append_quant: quantise new cache rows and scatter them to their slots.
//
// "DeepSeek-V4 KV Cache 深度分析", §二 (code evidence): the first 448 dims of
// the 512-d latent are quantised to FP8 and the last 64 (RoPE) dims stay
// BF16; §四: indexer keys may be Hadamard-rotated before their FP4
// quantisation (CKV_FMT_FP4H, hadamard.cuh).  "V4.1-Flash 공개", 핵심 내용, and "KV cache 890 bajtów na token",
// "Trzy mechanizmy": FP4 E2M1 values with one E4M3 scale per 16 channels,
// no global scale.
//
// One warp per row.  For 512-d rows each lane owns 16 consecutive channels
// (one FP4 block, or a 16-channel slice of the FP8 nope part); for 128-d rows
// each lane owns 4 channels and four lanes form an FP4 block.  Loads and stores
// are 8- to 32-byte vectors; the whole call is a few microseconds of launch
// latency for the row counts of a decode step.

#include <cstring>

#include "common.cuh"
#include "hadamard.cuh"

namespace ckv {

struct AppendArgs {
  uint8_t* data;
  void* scale;
  const __nv_bfloat16* src;
  const int64_t* slot;
  int64_t n_slots;  // batch * cap
  int32_t n;
  int32_t fmt, dim, nope_block;
  DevStatus* st;
};

__device__ __forceinline__ void load_bf16x16(const __nv_bfloat16* p, float (&v)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 a = q[0], b = q[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Up to kMaxAppendPlanes appends in one launch: plane k takes blocks
// [block0[k], block0[k + 1]), four rows per block.
constexpr int kMaxAppendPlanes = CKV_APPEND_MAX_PLANES;
struct AppendBatch {
  AppendArgs p[kMaxAppendPlanes];
  int32_t block0[kMaxAppendPlanes + 1];
  int32_t n_planes;
};

// Row `row` of append `a`, by one warp.
__device__ __forceinline__ void append_row(const AppendArgs& a, int row, int lane) {
  if (row >= a.n) return;
  const int64_t slot = a.slot[row];
  if (slot < 0) return;
  if (slot >= a.n_slots) {
    if (lane == 0) report(a.st, CKV_ERR_DEVICE_BOUNDS, row);
    return;
  }
  const __nv_bfloat16* src = a.src + (int64_t)row * a.dim;

  if (a.dim == 512) {
    float v[16];
    load_bf16x16(src + lane * 16, v);
    if (a.fmt == CKV_FMT_BF16) {
      const uint4* s = reinterpret_cast<const uint4*>(src + lane * 16);
      uint4* d = reinterpret_cast<uint4*>(a.data + slot * 1024 + lane * 32);
      d[0] = s[0];
      d[1] = s[1];
    } else if (a.fmt == CKV_FMT_FP4) {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const uint8_t sc = e4m3_code(__fdiv_rn(amax, 6.0f));
      const float s = e4m3_value(sc);
      uint32_t lo = 0, hi = 0;
      if (s > 0.f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) lo |= e2m1_code(__fdiv_rn(v[i], s)) << (4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) hi |= e2m1_code(__fdiv_rn(v[8 + i], s)) << (4 * i);
      }
      *reinterpret_cast<uint2*>(a.data + slot * 256 + lane * 8) = make_uint2(lo, hi);
      reinterpret_cast<uint8_t*>(a.scale)[slot * 32 + lane] = s > 0.f ? sc : (uint8_t)0;
    } else {  // CKV_FMT_MIXED: lanes 0..27 nope, 28..31 rope
      const bool nope = lane < 28;
      float amax = 0.f;
      if (nope) {
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
      }
      // block reduction: block 448 -> all 28 nope lanes; block 64 -> 4 lanes
      if (a.nope_block == 448) {
        amax = warp_max(amax);
      } else {
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      }
      uint8_t* entry = a.data + slot * 576;
      if (nope) {
        const float s = __fdiv_rn(amax, 448.0f);
        uint32_t w[4] = {0, 0, 0, 0};
        if (s > 0.f) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i >> 2] |= (uint32_t)e4m3_code(__fdiv_rn(v[i], s)) << (8 * (i & 3));
        }
        *reinterpret_cast<uint4*>(entry + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        const int nblk = 448 / a.nope_block;
        const int lanes_per_blk = a.nope_block / 16;
        if (lane % lanes_per_blk == 0)
          reinterpret_cast<float*>(a.scale)[slot * nblk + lane / lanes_per_blk] = s;
      } else {
        const uint4* s = reinterpret_cast<const uint4*>(src + lane * 16);
        uint4* d = reinterpret_cast<uint4*>(entry + 448 + (lane - 28) * 32);
        d[0] = s[0];
        d[1] = s[1];
      }
    }
  } else {  // dim 128: 4 channels per lane
    const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * 4);
    if (a.fmt == CKV_FMT_BF16) {
      *reinterpret_cast<uint2*>(a.data + slot * 256 + lane * 8) = raw;
    } else {  // CKV_FMT_FP4 / CKV_FMT_FP4H (the latter rotated first)
      float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                    __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
      if (a.fmt == CKV_FMT_FP4H) hadamard128_warp(v, lane);
      uint8_t sc;
      const uint32_t c = fp4_quant_lane4(v, sc);
      *reinterpret_cast<uint16_t*>(a.data + slot * 64 + lane * 2) = (uint16_t)c;
      if ((lane & 3) == 0) reinterpret_cast<uint8_t*>(a.scale)[slot * 8 + (lane >> 2)] = sc;
    }
  }
}

__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ AppendBatch b) {
  pdl_wait();
  pdl_launch_dependents();
  int k = 0;
  while (k + 1 < b.n_planes && (int)blockIdx.x >= b.block0[k + 1]) ++k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  append_row(b.p[k], ((int)blockIdx.x - b.block0[k]) * 4 + warp, lane);
}

cudaError_t launch_append_multi(const ckv_plane* p, const void* const* src, const int64_t* const* slot,
                                const int32_t* n, int n_planes, DevStatus* st, cudaStream_t stream) {
  if (n_planes < 1 || n_planes > kMaxAppendPlanes) return cudaErrorInvalidValue;
  AppendBatch b;
  memset(&b, 0, sizeof(b));
  int blocks = 0;
  for (int k = 0; k < n_planes; ++k) {
    AppendArgs& a = b.p[k];
    a.data = static_cast<uint8_t*>(p[k].data);
    a.scale = p[k].scale;
    a.src = static_cast<const __nv_bfloat16*>(src[k]);
    a.slot = slot[k];
    a.n_slots = plane_rows(p[k]);
    a.n = n[k];
    a.fmt = p[k].fmt;
    a.dim = p[k].dim;
    a.nope_block = p[k].nope_block;
    a.st = st;
    b.block0[k] = blocks;
    blocks += (n[k] + 3) / 4;
  }
  b.block0[n_planes] = blocks;
  b.n_planes = n_planes;
  if (blocks == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute at[1] = {pdl_attribute()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel, b);
}

cudaError_t launch_append(const ckv_plane& p, const void* src, const int64_t* slot, int32_t n,
                          DevStatus* st, cudaStream_t stream) {
  return launch_append_multi(&p, &src, &slot, &n, 1, st, stream);
}

}  // namespace ckv

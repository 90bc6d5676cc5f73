// Hadamard rotation + FP4 block quantisation of a 128-d indexer vector held
// by one warp (4 channels per lane).
//
// "DeepSeek-V4 KV Cache 深度分析", §四: the indexer's FP4 quantisation is a
// Hadamard rotation followed by the FP4 quantiser over all 128 dims.  The
// rotation is the Sylvester-ordered Hadamard matrix of order 128 scaled by
// 1/sqrt(128), computed as the fast Walsh-Hadamard transform in f32: stage
// h = 1, 2, 4, ..., 64 turns every pair (j, j + h) with bit h of j clear into
// (a + b, a - b).  Channel j = 4 * lane + m; stages 1 and 2 pair channels of
// one lane, stages 4 .. 64 pair lane l with lane l ^ (h / 4).  Each output is
// the same chain of f32 additions in the same order as the canonical
// transform, so the values (and the quantised bytes) do not depend on how the
// channels are spread over threads.
#pragma once

#include "common.cuh"

namespace ckv {

// fl32(1 / sqrt(128)) = fl32(sqrt(2)) / 16
constexpr uint32_t kInvSqrt128Bits = 0x3DB504F3u;

// In-place rotation of the warp's 128 channels (v[m] = channel 4 * lane + m).
__device__ __forceinline__ void hadamard128_warp(float (&v)[4], int lane) {
  float t0 = v[0] + v[1], t1 = v[0] - v[1], t2 = v[2] + v[3], t3 = v[2] - v[3];   // h = 1
  v[0] = t0 + t2;                                                                  // h = 2
  v[2] = t0 - t2;
  v[1] = t1 + t3;
  v[3] = t1 - t3;
#pragma unroll
  for (int x = 1; x <= 16; x <<= 1) {   // h = 4x: partner lane ^ x
    const bool upper = (lane & x) != 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float p = __shfl_xor_sync(0xffffffffu, v[m], x);
      v[m] = upper ? p - v[m] : v[m] + p;
    }
  }
  const float sc = __uint_as_float(kInvSqrt128Bits);
#pragma unroll
  for (int m = 0; m < 4; ++m) v[m] = v[m] * sc;
}

// FP4 block quantisation of the warp's 128 channels (4 per lane, four lanes
// per 16-channel block): E4M3 scale of amax / 6, E2M1 codes of x / scale, sign
// of zero kept, a zero scale gives zero codes.  Returns the lane's two code
// bytes (channel 4l in the low nibble) and sets `scale` (the block's scale
// code, the same in its four lanes).
__device__ __forceinline__ uint32_t fp4_quant_lane4(const float (&v)[4], uint8_t& scale) {
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const uint8_t sc = e4m3_code(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_value(sc);
  uint32_t c = 0;
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) c |= e2m1_code(__fdiv_rn(v[i], s)) << (4 * i);
  }
  scale = s > 0.f ? sc : (uint8_t)0;
  return c;
}

}  // namespace ckv

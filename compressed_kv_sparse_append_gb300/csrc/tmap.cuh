// Host-side encoding of 2-D TMA tensor maps, with a per-thread cache.
//
// A tensor map is a pure function of its encoding arguments, and a decode
// step encodes the same few maps (the same planes, the same boxes) on every
// call.  Each host thread keeps the last kTmapCacheSize maps it encoded and
// copies a hit instead of calling the driver again.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>

namespace ckv {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  // looked up once (a function-local static is initialised once, thread-safely)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

struct TmapKey {
  uint64_t data;
  uint64_t dims[2];
  uint64_t stride;
  uint32_t box[2];
  int32_t dtype, swizzle;
};

constexpr int kTmapCacheSize = 16;

// 2-D tiled map over `data` ([dims[1]] rows of dims[0] elements, row pitch
// `stride` bytes), element strides 1, no interleave, L2 promotion 256 B, no
// NaN fill.  Returns false if the driver rejects the arguments.
inline bool encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* data, uint64_t dim0,
                           uint64_t dim1, uint64_t stride, uint32_t box0, uint32_t box1,
                           CUtensorMapSwizzle sw) {
  TmapKey k;
  memset(&k, 0, sizeof(k));
  k.data = reinterpret_cast<uint64_t>(data);
  k.dims[0] = dim0;
  k.dims[1] = dim1;
  k.stride = stride;
  k.box[0] = box0;
  k.box[1] = box1;
  k.dtype = (int32_t)dt;
  k.swizzle = (int32_t)sw;
  struct Entry {
    TmapKey key;
    CUtensorMap map;
    bool valid;
  };
  thread_local Entry cache[kTmapCacheSize] = {};
  thread_local int next = 0;
  for (int i = 0; i < kTmapCacheSize; ++i)
    if (cache[i].valid && memcmp(&cache[i].key, &k, sizeof(k)) == 0) {
      *m = cache[i].map;
      return true;
    }
  auto enc = tmap_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {dim0, dim1};
  cuuint64_t strides[1] = {stride};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t es[2] = {1, 1};
  if (enc(m, dt, 2, const_cast<void*>(data), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& e = cache[next];
  next = (next + 1) % kTmapCacheSize;
  e.key = k;
  e.map = *m;
  e.valid = true;
  return true;
}

}  // namespace ckv

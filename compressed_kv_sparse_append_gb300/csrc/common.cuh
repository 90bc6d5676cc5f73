// Device helpers shared by the libckv kernels: status reporting, bounded
// mbarrier waits, tcgen05 (TMEM allocation, MMA, loads/stores), shared-memory
// matrix descriptors and cluster (DSMEM) access.  Everything is hand-written
// inline PTX for sm_103a.
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>

#include "../../include/ckv.h"

namespace ckv {

// ---- host: one-time setup per device, safe with several host threads ----
constexpr int kOnceDevices = 64;
struct DeviceOnce {
  std::once_flag flag[kOnceDevices];
  cudaError_t err[kOnceDevices] = {};
};
// Runs f() (returning cudaError_t) once for the current device; every later
// call, from any thread, returns that first result.
template <class F>
inline cudaError_t once_per_device(DeviceOnce& o, F&& f) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kOnceDevices) return cudaErrorInvalidDevice;
  std::call_once(o.flag[dev], [&] { o.err[dev] = f(dev); });
  return o.err[dev];
}


// Rows of a plane's data (and scale) arrays: batch * cap when dense,
// n_pages * page_size when paged.
inline int64_t plane_rows(const ckv_plane& p) {
  return p.block_table ? (int64_t)p.n_pages * p.page_size : (int64_t)p.batch * p.cap;
}

// Row of entry `pos` of sequence b in a plane (dense: b * cap + pos; paged:
// through the block table, bt_cols = cap / page_size entries per sequence).
__device__ __forceinline__ int64_t plane_row(const int32_t* bt, int page, int bt_cols, int64_t cap,
                                             int b, int64_t pos) {
  if (!bt) return (int64_t)b * cap + pos;
  const int pg = __ldg(bt + (int64_t)b * bt_cols + (int)(pos / page));
  return (int64_t)pg * page + pos % page;
}

// ------------------------------------------------------------ status ----
// The first 256 bytes of every workspace: [0] sticky error code (the most
// recent nonzero one), [1] count of events, [2] detail (index, stage...).
struct DevStatus {
  int32_t code;
  uint32_t count;
  int32_t detail;
  int32_t pad[61];
};
static_assert(sizeof(DevStatus) == 256, "status block is 256 bytes");

static __device__ __noinline__ void report(DevStatus* st, int32_t code, int32_t detail) {
  if (st == nullptr) return;
  atomicExch(&st->code, code);
  atomicAdd(&st->count, 1u);
  atomicExch(&st->detail, detail);
}

// Limits of every spin-wait in the kernels: wall clock, SM cycles and
// iterations -- whichever expires first ends the wait, so a wait ends even if
// one of the clocks does not advance.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr long long kWaitLimitCycles = 4000000000ll;
constexpr uint32_t kWaitLimitIters = 1u << 24;

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Arrive on the barrier at `remote` (a shared::cluster address of a CTA in
// the cluster), releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// CTA-scope variants for kernels launched without clusters: every arrival
// comes from this CTA (or its own async operations), so the acquire need not
// reach cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cta(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The bounded loop behind every wait below.
// kind 0: try_wait, acquire at cluster scope; 1: try_wait, CTA scope;
// 2: polling test_wait, cluster scope.
static __device__ __forceinline__ bool mbar_wait_slow(uint32_t a, uint32_t parity, DevStatus* st,
                                            volatile int* abort, int where, uint64_t limit_ns,
                                            int kind) {
  const uint64_t t0 = globaltimer();
  const long long c0 = clock64();
  const uint32_t mask = kind == 2 ? 255u : 63u;
  const uint32_t max_it = kind == 2 ? 16u * kWaitLimitIters : kWaitLimitIters;
  for (uint32_t it = 1;; ++it) {
    const bool ok = kind == 0 ? mbar_try_wait(a, parity)
                              : kind == 1 ? mbar_try_wait_cta(a, parity) : mbar_test_wait(a, parity);
    if (ok) return true;
    if ((it & mask) == 0) {
      if (*abort) return false;
      if (it >= max_it || clock64() - c0 > kWaitLimitCycles || globaltimer() - t0 > limit_ns) {
        report(st, CKV_ERR_TIMEOUT, where);
        *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool mbar_test_wait_cta(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// A phase that has already completed passes on a non-suspending test; only
// an open one takes the (suspending) bounded wait.
__device__ __forceinline__ bool mbar_wait_cta(uint64_t* bar, uint32_t parity, DevStatus* st,
                                              volatile int* abort, int where,
                                              uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test_wait_cta(a, parity)) return true;
  return mbar_wait_slow(a, parity, st, abort, where, limit_ns, 1);
}

// Bounded polling wait (non-suspending test_wait) for barriers whose
// arrivals come from other CTAs of the cluster.
__device__ __forceinline__ bool mbar_wait_poll(uint64_t* bar, uint32_t parity, DevStatus* st,
                                               volatile int* abort, int where,
                                               uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test_wait(a, parity)) return true;
  return mbar_wait_slow(a, parity, st, abort, where, limit_ns, 2);
}

// Bounded wait for the phase with parity `parity` to complete.  On expiry
// it records CKV_ERR_TIMEOUT (detail = `where`), raises *abort and returns
// false; once *abort is set every later wait returns false at once.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, DevStatus* st,
                                          volatile int* abort, int where,
                                          uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  return mbar_wait_slow(a, parity, st, abort, where, limit_ns, 0);
}

// Bounded spin of one thread until the global counter *cnt reaches
// `target` (acquire at GPU scope, so the writes released before each
// increment are visible once it returns true).  On expiry it records
// CKV_ERR_TIMEOUT (detail = `where`), raises *abort and returns false.
__device__ __forceinline__ bool spin_until_geq(const uint32_t* cnt, uint32_t target, DevStatus* st,
                                               volatile int* abort, int where,
                                               uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t g0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    if (*abort || it >= kWaitLimitIters || globaltimer() - g0 > limit_ns) {
      if (!*abort) report(st, CKV_ERR_TIMEOUT, where);
      *abort = 1;
      return false;
    }
    __nanosleep(64);
  }
}

// Optional progress counters (debugging): slot k of the status block's
// spare words counts events of kind k.  Enabled per launch.
static __device__ __noinline__ void progress_add(DevStatus* st, int k) {
  if (st != nullptr) atomicAdd(reinterpret_cast<unsigned int*>(&st->pad[k]), 1u);
}
__device__ __forceinline__ void progress(DevStatus* st, bool on, int k) {
  if (on) progress_add(st, k);
}

// Debug timeline: store the clock64 offset of an event in spare word `slot`
// of the status block.
static __device__ __noinline__ void trace_at_store(DevStatus* st, int slot, long long t0) {
  if (st != nullptr && slot >= 0 && slot < 61) st->pad[slot] = (int32_t)(clock64() - t0);
}
__device__ __forceinline__ void trace_at(DevStatus* st, bool on, int slot, long long t0) {
  if (on) trace_at_store(st, slot, t0);
}

// Asynchronous global -> shared copies (cp.async): 16 bytes through L2
// only, or 4 bytes cached in L1; the caller waits with cp.async.wait_all /
// wait_group.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4_ca(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Launch attribute for programmatic stream serialisation (host side).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  return at;
}

// -------------------------------------- programmatic dependent launch ----
// Every kernel is launched with programmatic stream serialisation, so it may
// start while the previous kernel in the stream is finishing.  pdl_wait()
// blocks until the grids this one depends on have completed and their
// memory operations are visible; each kernel calls it before it reads or
// writes anything in global memory.  pdl_launch_dependents() lets the next
// kernel begin launching (it still waits in its own pdl_wait()).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- fences ----
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------- cluster ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of `local` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ------------------------------------------------------------- tcgen05 ----
__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), kind::f16 (bf16 in, f32 acc).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled FP4 (E2M1 x E2M1, one UE4M3 scale per 16 K-elements).
__device__ __forceinline__ void umma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// All previously issued tcgen05.mma of this thread arrive on `bar` when done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread l of the warp gets row
// (lane base + l), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31]));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a),
               "r"(b), "r"(c), "r"(d));
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), descriptor version 1, swizzle mode.
//   swizzle: 0 none, 2 = 128B, 4 = 64B, 6 = 32B.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7) << 61;
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, f32 accumulator.
//   a_mn / b_mn: 1 when that operand is MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::mxf4nvf4 block-scaled: E2M1 A and B (format
// code 1), UE4M3 scales (scale-type bit 0), scale-factor ids 0, K-major.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------- number formats ----
__device__ __forceinline__ uint8_t e4m3_code(float x) {
  uint8_t c = (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
  // Codes carry the sign of x, also when the magnitude rounds to zero.
  if (signbit(x)) c |= 0x80;
  return c;
}
__device__ __forceinline__ float e4m3_value(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}
__device__ __forceinline__ uint32_t e2m1_code(float x) {
  uint32_t c = (uint32_t)__nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest) & 0xF;
  if (signbit(x)) c |= 0x8;
  return c;
}
// E2M1 magnitude table: {0, .5, 1, 1.5, 2, 3, 4, 6} (1 sign, 2 exponent
// bits with bias 1, 1 mantissa bit).
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float v = (e == 0) ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
  return (c & 8u) ? -v : v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Order-preserving map of an f32 score to u32 (larger score -> larger key);
// -0.0 is first turned into +0.0.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s == 0.0f ? 0.0f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

}  // namespace ckv

// Host side of the libckv C ABI: argument validation, workspace layout,
// kernel dispatch and the CSA2 group driver.  Every check runs before any
// work is enqueued; nothing here allocates device memory.

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "indexer.cuh"
#include "attention.cuh"

namespace ckv {
cudaError_t launch_append(const ckv_plane& p, const void* src, const int64_t* slot, int32_t n,
                          DevStatus* st, cudaStream_t stream);
cudaError_t launch_append_multi(const ckv_plane* p, const void* const* src, const int64_t* const* slot,
                                const int32_t* n, int n_planes, DevStatus* st, cudaStream_t stream);
}

namespace ckv {

// Makes one bounded wait of the kinds the kernels use run out: mode 0 an
// mbarrier phase that nothing completes (the pipeline waits), mode 1 a
// global counter that nothing increments (the cross-CTA merge wait).  The
// wait records CKV_ERR_TIMEOUT in the status block after `limit_ns` and the
// kernel returns; nothing else is touched.
__global__ void wait_probe_kernel(DevStatus* st, const uint32_t* never_set, int mode, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (mode == 0) mbar_wait(&bar, 0, st, &abort_flag, 90, limit_ns);
    else spin_until_geq(never_set, 1u, st, &abort_flag, 91, limit_ns);
  }
  __syncthreads();
}

}  // namespace ckv

using namespace ckv;

namespace {

constexpr size_t kStatusBytes = 256;

// An NVTX range named after the entry point around each call's host work
// (validation and enqueue), so that a timeline tool shows which library call
// issued which launches.  Without a tool attached each push/pop is a test of
// an unset function pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates a plane of the given dim for `B` sequences.
ckv_status check_plane(const ckv_plane* p, int dim, int B) {
  if (!p || !p->data || !aligned16(p->data)) return CKV_ERR_INVALID;
  if (p->dim != dim || p->cap <= 0 || p->batch < B) return CKV_ERR_INVALID;
  if (p->block_table) {
    // paged: whole pages of a multiple of 128 rows, a cap of whole pages,
    // row numbers that fit int32 (TMA coordinates)
    if (p->page_size <= 0 || p->page_size % 128 != 0 || p->n_pages <= 0) return CKV_ERR_INVALID;
    if (p->cap % p->page_size != 0) return CKV_ERR_INVALID;
    if ((int64_t)p->n_pages * p->page_size >= ((int64_t)1 << 31)) return CKV_ERR_UNSUPPORTED;
  }
  if (p->fmt == CKV_FMT_BF16) return CKV_OK;
  if (p->fmt == CKV_FMT_FP4) {
    if (!p->scale || (dim != 512 && dim != 128)) return CKV_ERR_INVALID;
    return CKV_OK;
  }
  if (p->fmt == CKV_FMT_FP4H) {   // Hadamard-rotated FP4: indexer keys only
    if (dim != 128) return CKV_ERR_UNSUPPORTED;
    if (!p->scale) return CKV_ERR_INVALID;
    return CKV_OK;
  }
  if (p->fmt == CKV_FMT_MIXED) {
    if (dim != 512) return CKV_ERR_UNSUPPORTED;
    if (!p->scale || !aligned16(p->scale)) return CKV_ERR_INVALID;
    if (p->nope_block != 448 && p->nope_block != 64) return CKV_ERR_UNSUPPORTED;
    return CKV_OK;
  }
  return CKV_ERR_INVALID;
}

struct IndexLayout {
  int chunk, n_chunks;
  size_t seq_off, hist_off, count_off, key_off, idx_off, bytes;  // relative to the index region
};

// Between-call state of the single-op calls, at fixed offsets after the
// status block, so that index/top-k and attention calls with the same B may
// share one workspace: every op's scratch starts after all of it.
//   [0, index_zero_bytes)   index: per-sequence state (merge ticket, the
//                           range of histogram bins in use), then the
//                           per-sequence 8192-bin key histograms
//   [.., + attn_zero_bytes) attention: per-sequence, per-half merge counters
// Each op leaves its own part zero when it finishes.
size_t index_zero_bytes(int B) {
  return align_up((size_t)B * kSeqWords * 4, 256) + (size_t)B * kBins * 4;
}
size_t attn_zero_bytes(int B) { return align_up((size_t)B * 2 * sizeof(uint32_t), 256); }
size_t shared_zero_bytes(int B) { return index_zero_bytes(B) + attn_zero_bytes(B); }

// Chunking of one index pass and the scratch after the shared state: per
// chunk its candidate count and real-key count, then candidate keys and
// entries (one slot per entry of the chunk, the most a chunk can keep).
IndexLayout index_layout(int B, int n_comp_max, bool pool_mode, int pool_len) {
  IndexLayout L;
  if (pool_mode) {
    L.chunk = 256;
    L.n_chunks = (pool_len + 255) / 256;
    if (L.n_chunks < 1) L.n_chunks = 1;
  } else {
    const int64_t total = (int64_t)B * n_comp_max;
    int64_t per = (total + 151) / 152;
    int c = (int)align_up((size_t)per, 256);
    c = c < 1024 ? 1024 : c;
    c = c > kMaxChunk ? kMaxChunk : c;
    L.chunk = c;
    L.n_chunks = (n_comp_max + c - 1) / c;
    if (L.n_chunks < 1) L.n_chunks = 1;
  }
  L.seq_off = 0;
  L.hist_off = align_up((size_t)B * kSeqWords * 4, 256);
  L.count_off = shared_zero_bytes(B);   // scratch after the attention's counters too
  const size_t cand = (size_t)B * L.n_chunks * L.chunk * 4;
  L.key_off = L.count_off + align_up((size_t)B * L.n_chunks * 8, 256);
  L.idx_off = L.key_off + align_up(cand, 256);
  L.bytes = L.idx_off + align_up(cand, 256);
  return L;
}

ckv_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return CKV_ERR_WORKSPACE;
  if (ws_bytes < need) return CKV_ERR_WORKSPACE;
  return CKV_OK;
}

// FP4 keys are scored on the block-scaled tensor cores; CKV_INDEXER=simt in
// the environment selects the CUDA-core scorer (used to cross-check them).
bool use_umma_indexer() {
  static const bool v = [] {
    const char* e = getenv("CKV_INDEXER");
    return !(e && strcmp(e, "simt") == 0);
  }();
  return v;
}

// CKV_DEBUG_PROGRESS (1 .. 6; read once per process) turns on the
// kernels' debugging records in the status block.
int debug_progress() {
  static const int v = [] {
    const char* e = getenv("CKV_DEBUG_PROGRESS");
    return (e && e[0] >= '1' && e[0] <= '6') ? e[0] - '0' : 0;
  }();
  return v;
}

ckv_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CKV_OK;
  (void)cudaGetLastError();
  return CKV_ERR_CUDA;
}

// Enqueues one index/top-k pass; `region` is the index scratch.
ckv_status run_index(const ckv_plane* keys, const int32_t* n_comp, int B, int n_comp_max,
                     const void* q_idx, const float* w, int HI, int topk, const int32_t* pool,
                     int pool_len, int32_t* out_idx, int32_t* out_pool, int pool_out, float* dbg,
                     DevStatus* st, uint8_t* region, cudaStream_t stream) {
  IndexLayout L = index_layout(B, n_comp_max, pool != nullptr, pool_len);
  IndexArgs a;
  a.kdata = static_cast<const uint8_t*>(keys->data);
  a.kscale = static_cast<const uint8_t*>(keys->scale);
  a.cap = keys->cap;
  a.bt = keys->block_table;
  a.page = keys->block_table ? keys->page_size : 0;
  a.bt_cols = keys->block_table ? (int)(keys->cap / keys->page_size) : 0;
  a.rows = plane_rows(*keys);
  a.fmt = keys->fmt;
  a.n_comp = n_comp;
  a.B = B;
  a.n_comp_max = n_comp_max;
  a.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  a.w = w;
  a.HI = HI;
  a.pool = pool;
  a.pool_len = pool_len;
  a.topk = topk;
  a.pool_out = out_pool ? pool_out : 0;
  a.chunk = L.chunk;
  a.n_chunks = L.n_chunks;
  a.seq_state = reinterpret_cast<uint32_t*>(region + L.seq_off);
  a.ghist = reinterpret_cast<uint32_t*>(region + L.hist_off);
  a.ccount = reinterpret_cast<uint32_t*>(region + L.count_off);
  a.cand_key = reinterpret_cast<uint32_t*>(region + L.key_off);
  a.cand_idx = reinterpret_cast<int32_t*>(region + L.idx_off);
  a.out_idx = out_idx;
  a.out_pool = out_pool;
  a.dbg = dbg;
  a.st = st;
  a.trace = debug_progress() == 2 ? 1 : 0;
  const int64_t rows = plane_rows(*keys);
  if (use_umma_indexer() && index_umma_supported(a, rows))
    return cuda_status(launch_index_umma(a, rows, stream));
  return cuda_status(launch_index_simt(a, stream));
}

ckv_status check_index_args(const ckv_plane* keys, const int32_t* n_comp, int B, int n_comp_max,
                            const void* q_idx, const float* w, int HI, int topk,
                            const int32_t* pool, int pool_len, const int32_t* out_idx,
                            const int32_t* out_pool, int pool_out) {
  if (B <= 0 || !n_comp || !q_idx || !w || !out_idx) return CKV_ERR_INVALID;
  if (!aligned16(q_idx)) return CKV_ERR_INVALID;
  ckv_status s = check_plane(keys, 128, B);
  if (s) return s;
  if (keys->fmt != CKV_FMT_FP4 && keys->fmt != CKV_FMT_FP4H && keys->fmt != CKV_FMT_BF16)
    return CKV_ERR_UNSUPPORTED;
  if (HI <= 0 || HI > kMaxHI) return CKV_ERR_UNSUPPORTED;
  if (n_comp_max < 0 || n_comp_max > keys->cap) return CKV_ERR_INVALID;
  if (topk <= 0 || topk > kMaxPool) return CKV_ERR_UNSUPPORTED;
  if (index_layout(B, n_comp_max, pool != nullptr, pool_len).n_chunks > kMaxChunksPerSeq)
    return CKV_ERR_UNSUPPORTED;
  if (pool) {
    if (out_pool || pool_len <= 0 || pool_len > kMaxChunk) return CKV_ERR_INVALID;
  }
  if (out_pool && (pool_out < topk || pool_out > kMaxPool)) return CKV_ERR_INVALID;
  return CKV_OK;
}

// Scratch of one index pass; a pool-mode pass chunks the pool.
size_t index_ws_bytes(int B, int n_comp_max, bool pool_mode, int pool_len) {
  return index_layout(B, n_comp_max, pool_mode, pool_len).bytes;
}

// The attention's split-KV merge state: the partials of up to 2 * kMaxPairs
// CTAs per sequence and layer (kPartFloats floats each), then one counter per
// sequence, layer and half (the merge ticket).
size_t attn_part_bytes(int B, int layers) {
  return align_up((size_t)layers * B * 2 * kMaxPairs * kPartFloats * sizeof(float), 256);
}
size_t attn_ws_bytes(int B, int layers) {
  return attn_part_bytes(B, layers) + align_up((size_t)layers * B * 2 * sizeof(uint32_t), 256);
}
// Layers [l0, ...) of a region sized for `layers`: their partials and
// counters follow those of layers 0 .. l0 - 1 (inside, a launch indexes them
// by its own grid z).
void attn_set_ws(AttnArgs& a, uint8_t* region, int B, int layers, int l0 = 0) {
  a.part = reinterpret_cast<float*>(region) + (size_t)l0 * B * 2 * kMaxPairs * kPartFloats;
  a.tickets = reinterpret_cast<uint32_t*>(region + attn_part_bytes(B, layers)) + (size_t)l0 * B * 2;
}
// The single-op attention calls: counters in their fixed slot of the shared
// layout, partials after it.
size_t attn_single_ws_bytes(int B) { return shared_zero_bytes(B) + attn_part_bytes(B, 1); }
void attn_set_ws_single(AttnArgs& a, uint8_t* region, int B) {
  a.tickets = reinterpret_cast<uint32_t*>(region + index_zero_bytes(B));
  a.part = reinterpret_cast<float*>(region + shared_zero_bytes(B));
}

// Picks the number of CTA pairs per sequence and the cluster shape; each
// pair keeps at least two 64-row tiles.  A cluster of all 2G CTAs of a
// sequence merges after a hardware-scheduled cluster barrier.  Pair clusters
// fit more pairs on the GPU; their sequence's partials are merged by the
// last CTA of each half to finish (a counter in the workspace, no waiting),
// and they are taken when they leave the busiest pair fewer tiles.  Neither
// needs more than the launch's clusters resident at once.
struct PairChoice {
  int G;
  int cluster_all;
};
PairChoice choose_pairs(int n_seq, int n_rows_max) {
  const int tiles = (n_rows_max + 63) / 64;
  int g_all = 1, g_pair = 1;
  const int fit2 = attn_max_active_clusters(2);
  for (int G = 2; G <= kMaxPairs && tiles >= 2 * G; ++G) {
    const int fit = attn_max_active_clusters(2 * G);
    if (fit > 0 && n_seq <= fit) g_all = G;
    if (fit2 > 0 && n_seq * G <= fit2) g_pair = G;
  }
  // fewer tiles for the busiest pair wins; on a tie the sequence-wide
  // clusters, whose merge every CTA shares (with pair clusters one CTA per
  // half merges all G partials)
  const int t_all = (tiles + g_all - 1) / g_all, t_pair = (tiles + g_pair - 1) / g_pair;
  return t_pair < t_all ? PairChoice{g_pair, 0} : PairChoice{g_all, 1};
}

ckv_status check_attn_common(const ckv_plane* kv, const ckv_plane* win, const int32_t* win_len,
                             int B, const void* q, int H, void* out, float sm_scale) {
  if (B <= 0 || !win_len || !q || !out || !aligned16(q) || !aligned16(out)) return CKV_ERR_INVALID;
  if (!(sm_scale > 0.f) || !(sm_scale < INFINITY)) return CKV_ERR_INVALID;
  if (H <= 0 || H > kMaxHeads) return CKV_ERR_UNSUPPORTED;
  ckv_status s = check_plane(kv, 512, B);
  if (s) return s;
  s = check_plane(win, 512, B);
  if (s) return s;
  if (win->fmt != kv->fmt || (kv->fmt == CKV_FMT_MIXED && win->nope_block != kv->nope_block))
    return CKV_ERR_INVALID;
  if (win->block_table) return CKV_ERR_UNSUPPORTED;   // window rings are dense
  return CKV_OK;
}

AttnArgs attn_args(const ckv_plane* kv, const ckv_plane* win, const int32_t* win_len,
                   const void* q, int H, float sm_scale, void* out, float* lse, DevStatus* st) {
  AttnArgs a;
  a.kv_data = static_cast<const uint8_t*>(kv->data);
  a.kv_scale = kv->scale;
  a.kv_cap = kv->cap;
  a.kv_rows = plane_rows(*kv);
  a.kv_bt = kv->block_table;
  a.kv_page = kv->block_table ? kv->page_size : 0;
  a.kv_bt_cols = kv->block_table ? (int)(kv->cap / kv->page_size) : 0;
  a.win_data = static_cast<const uint8_t*>(win->data);
  a.win_scale = win->scale;
  a.win_cap = win->cap;
  a.fmt = kv->fmt;
  a.nope_block = kv->nope_block;
  a.idx = nullptr;
  a.topk = 0;
  a.n_comp = nullptr;
  a.n_comp_max = 0;
  a.win_len = win_len;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.H = H;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.G = 1;
  a.cluster_all = 1;
  a.part = nullptr;
  a.tickets = nullptr;
  a.st = st;
  a.use_tma = 0;
  a.progress = debug_progress();
  a.rope_pos = nullptr;
  a.rope_freq = nullptr;
  a.rope_q = 0;
  a.rope_out = 0;
  return a;
}

// RoPE of the attention's ends: a null descriptor or pos means none.
ckv_status set_rope(AttnArgs& a, const ckv_rope* r) {
  if (!r || !r->pos) return CKV_OK;
  if (!r->inv_freq) return CKV_ERR_INVALID;
  a.rope_pos = r->pos;
  a.rope_freq = r->inv_freq;
  a.rope_q = r->rotate_q ? 1 : 0;
  a.rope_out = r->rotate_out ? 1 : 0;
  return CKV_OK;
}

}  // namespace

extern "C" {

size_t ckv_workspace_bytes(int32_t op, int32_t B, int32_t H, int32_t HI, int32_t n_comp_max,
                           int32_t topk, int32_t pool_len) {
  (void)H;
  (void)HI;
  if (B <= 0) return kStatusBytes;
  switch (op) {
    case CKV_OP_INDEX_TOPK:
      // pool_len here: the pool_out of a CSA2 Full pass (0 for none); a
      // pool-mode (Reindex) pass never needs more than a full pass.
      return kStatusBytes +
             index_ws_bytes(B, n_comp_max, false, 0);
    case CKV_OP_CSA2: {
      size_t full = index_ws_bytes(B, n_comp_max, false, 0);
      size_t re = index_ws_bytes(B, n_comp_max, true, pool_len);
      size_t idx_region = align_up(full > re ? full : re, 256);
      size_t pool = align_up((size_t)B * (pool_len > 0 ? pool_len : 1) * 4, 256);
      size_t idxbuf = align_up((size_t)CKV_CSA2_MAX_LAYERS * B * topk * 4, 256);
      return kStatusBytes + idx_region + pool + idxbuf + attn_ws_bytes(B, CKV_CSA2_MAX_LAYERS);
    }
    case CKV_OP_SPARSE_ATTN:
    case CKV_OP_HCA_ATTN:
      return kStatusBytes + attn_single_ws_bytes(B);
    default:
      return kStatusBytes;
  }
}

ckv_status ckv_kv_append_quant(const ckv_plane* dst, const void* src_bf16, const int64_t* slot,
                               int32_t n, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("ckv_kv_append_quant");
  if (n < 0) return CKV_ERR_INVALID;
  if (!dst) return CKV_ERR_INVALID;
  ckv_status s = check_plane(dst, dst->dim, 1);
  if (s) return s;
  if (dst->dim != 512 && dst->dim != 128) return CKV_ERR_UNSUPPORTED;
  if (n > 0 && (!src_bf16 || !slot || !aligned16(src_bf16))) return CKV_ERR_INVALID;
  s = check_ws(ws, ws_bytes, kStatusBytes);
  if (s) return s;
  return cuda_status(launch_append(*dst, src_bf16, slot, n, static_cast<DevStatus*>(ws),
                                   static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_kv_append_quant_multi(const ckv_plane* dst, const void* const* src_bf16,
                                     const int64_t* const* slot, const int32_t* n, int32_t n_planes,
                                     void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("ckv_kv_append_quant_multi");
  if (!dst || !src_bf16 || !slot || !n || n_planes < 1 || n_planes > CKV_APPEND_MAX_PLANES)
    return CKV_ERR_INVALID;
  for (int k = 0; k < n_planes; ++k) {
    if (n[k] < 0) return CKV_ERR_INVALID;
    ckv_status s = check_plane(&dst[k], dst[k].dim, 1);
    if (s) return s;
    if (dst[k].dim != 512 && dst[k].dim != 128) return CKV_ERR_UNSUPPORTED;
    if (n[k] > 0 && (!src_bf16[k] || !slot[k] || !aligned16(src_bf16[k]))) return CKV_ERR_INVALID;
    // the planes' entry bytes must not overlap (rows land in no set order)
    for (int j = 0; j < k; ++j)
      if (dst[j].data == dst[k].data) return CKV_ERR_INVALID;
  }
  ckv_status s = check_ws(ws, ws_bytes, kStatusBytes);
  if (s) return s;
  return cuda_status(launch_append_multi(dst, src_bf16, slot, n, n_planes, static_cast<DevStatus*>(ws),
                                         static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_csa_index_topk(const ckv_plane* idx_keys, const int32_t* n_comp, int32_t B,
                              int32_t n_comp_max, const void* q_idx_bf16, const float* w,
                              int32_t HI, int32_t topk, const int32_t* pool, int32_t pool_len,
                              int32_t* out_idx, int32_t* out_pool, int32_t pool_out,
                              float* dbg_scores, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("ckv_csa_index_topk");
  ckv_status s = check_index_args(idx_keys, n_comp, B, n_comp_max, q_idx_bf16, w, HI, topk, pool,
                                  pool_len, out_idx, out_pool, pool_out);
  if (s) return s;
  const bool pool_mode = pool != nullptr;
  const size_t need = kStatusBytes + index_ws_bytes(B, n_comp_max, pool_mode, pool_mode ? pool_len : 0);
  s = check_ws(ws, ws_bytes, need);
  if (s) return s;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  return run_index(idx_keys, n_comp, B, n_comp_max, q_idx_bf16, w, HI, topk, pool, pool_len,
                   out_idx, out_pool, pool_out, dbg_scores, reinterpret_cast<DevStatus*>(w8),
                   w8 + kStatusBytes, static_cast<cudaStream_t>(stream));
}

ckv_status ckv_csa_sparse_attn_rope(const ckv_plane* kv, const ckv_plane* win, const int32_t* win_len,
                                    const int32_t* idx, int32_t B, int32_t topk, const void* q_bf16,
                                    int32_t H, float sm_scale, void* out_bf16, float* lse,
                                    const ckv_rope* rope, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("ckv_csa_sparse_attn");
  ckv_status s = check_attn_common(kv, win, win_len, B, q_bf16, H, out_bf16, sm_scale);
  if (s) return s;
  if (!idx || topk <= 0) return CKV_ERR_INVALID;
  if (topk > kMaxTopk) return CKV_ERR_UNSUPPORTED;
  s = check_ws(ws, ws_bytes, kStatusBytes + attn_single_ws_bytes(B));
  if (s) return s;
  AttnArgs a = attn_args(kv, win, win_len, q_bf16, H, sm_scale, out_bf16, lse,
                         static_cast<DevStatus*>(ws));
  s = set_rope(a, rope);
  if (s) return s;
  attn_set_ws_single(a, static_cast<uint8_t*>(ws) + kStatusBytes, B);
  a.idx = idx;
  a.topk = topk;
  const PairChoice pc = choose_pairs(B, topk + (int)win->cap);
  a.G = pc.G;
  a.cluster_all = pc.cluster_all;
  return cuda_status(launch_attention(a, B, static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_csa_sparse_attn(const ckv_plane* kv, const ckv_plane* win, const int32_t* win_len,
                               const int32_t* idx, int32_t B, int32_t topk, const void* q_bf16,
                               int32_t H, float sm_scale, void* out_bf16, float* lse, void* ws,
                               size_t ws_bytes, void* stream) {
  return ckv_csa_sparse_attn_rope(kv, win, win_len, idx, B, topk, q_bf16, H, sm_scale, out_bf16, lse,
                                  nullptr, ws, ws_bytes, stream);
}

ckv_status ckv_hca_attn_rope(const ckv_plane* kv, const int32_t* n_comp, int32_t n_comp_max,
                             const ckv_plane* win, const int32_t* win_len, int32_t B,
                             const void* q_bf16, int32_t H, float sm_scale, void* out_bf16,
                             float* lse, const ckv_rope* rope, void* ws, size_t ws_bytes,
                             void* stream) {
  NvtxRange nvtx_range("ckv_hca_attn");
  ckv_status s = check_attn_common(kv, win, win_len, B, q_bf16, H, out_bf16, sm_scale);
  if (s) return s;
  if (!n_comp || n_comp_max < 0 || n_comp_max > kv->cap) return CKV_ERR_INVALID;
  s = check_ws(ws, ws_bytes, kStatusBytes + attn_single_ws_bytes(B));
  if (s) return s;
  AttnArgs a = attn_args(kv, win, win_len, q_bf16, H, sm_scale, out_bf16, lse,
                         static_cast<DevStatus*>(ws));
  s = set_rope(a, rope);
  if (s) return s;
  attn_set_ws_single(a, static_cast<uint8_t*>(ws) + kStatusBytes, B);
  a.n_comp = n_comp;
  a.n_comp_max = n_comp_max;
  const PairChoice pc = choose_pairs(B, n_comp_max + (int)win->cap);
  a.G = pc.G;
  a.cluster_all = pc.cluster_all;
  return cuda_status(launch_attention(a, B, static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_hca_attn(const ckv_plane* kv, const int32_t* n_comp, int32_t n_comp_max,
                        const ckv_plane* win, const int32_t* win_len, int32_t B,
                        const void* q_bf16, int32_t H, float sm_scale, void* out_bf16,
                        float* lse, void* ws, size_t ws_bytes, void* stream) {
  return ckv_hca_attn_rope(kv, n_comp, n_comp_max, win, win_len, B, q_bf16, H, sm_scale, out_bf16,
                           lse, nullptr, ws, ws_bytes, stream);
}

// A side stream and two events per host thread and device, made on first
// use: the group call's first attention launch overlaps its Reindex passes.
struct SideResources {
  cudaStream_t s = nullptr;
  cudaEvent_t full = nullptr, re = nullptr;
};
cudaError_t side_resources(SideResources*& out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kOnceDevices) return cudaErrorInvalidDevice;
  static thread_local SideResources tl[kOnceDevices];
  SideResources& r = tl[dev];
  if (!r.s) {
    cudaStream_t s = nullptr;
    cudaEvent_t a = nullptr, b = nullptr;
    e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      if (b) cudaEventDestroy(b);
      if (a) cudaEventDestroy(a);
      if (s) cudaStreamDestroy(s);
      return e;
    }
    r.s = s;
    r.full = a;
    r.re = b;
  }
  out = &r;
  return cudaSuccess;
}

// The group's passes with one attention launch on the side stream: caller's
// stream: Full index (layer 0), the Reindex passes in layer order (the first
// of them launched beside the Full pass's tail by programmatic dependent
// launch), then the remaining layers' attention in launches of at most
// kLayersPerLaunch split evenly; side stream (after the Full pass): one
// attention launch of up to kLayersPerLaunch layers whose indices come from
// the Full pass, beside the Reindex passes.  root[l]: the layer whose index
// pass layer l uses.  The caller's stream finally waits for the side stream,
// so everything the call enqueues is ordered before its next work.
ckv_status csa2_group_overlapped(const ckv_csa2_group* g, const int* root, const int32_t* n_comp,
                                 int n_comp_max, const int32_t* win_len, int B, int H, int HI,
                                 int topk, float sm_scale, int pool_len, int32_t* idxbuf,
                                 int32_t* pool_buf, uint8_t* idx_region, uint8_t* attn_region,
                                 DevStatus* dst, cudaStream_t st) {
  const int L = g->n_layers;
  SideResources* side = nullptr;
  ckv_status s = cuda_status(side_resources(side));
  if (s) return s;
  int32_t* own[CKV_CSA2_MAX_LAYERS];
  for (int l = 0; l < L; ++l) own[l] = g->idx_out[l] ? g->idx_out[l] : idxbuf + (size_t)l * B * topk;
  // Full pass (layer 0) and the copies of the indices that reuse it
  s = run_index(&g->idx_keys, n_comp, B, n_comp_max, g->q_idx[0], g->w[0], HI, topk, nullptr, 0,
                own[0], pool_buf, pool_len, nullptr, dst, idx_region, st);
  if (s) return s;
  s = cuda_status(cudaEventRecord(side->full, st));
  if (s) return s;
  // Reindex passes on the caller's stream, the first attention launch on
  // the side stream once the Full pass is done
  s = cuda_status(cudaStreamWaitEvent(side->s, side->full, 0));
  if (s) return s;
  for (int l = 1; l < L; ++l)
    if (g->role[l] == CKV_CSA2_REINDEX) {
      s = run_index(&g->idx_keys, n_comp, B, n_comp_max, g->q_idx[l], g->w[l], HI, topk, pool_buf,
                    pool_len, own[l], nullptr, 0, nullptr, dst, idx_region, st);
      if (s) return s;
    }
  // launch order: the first kLayersPerLaunch Full-derived layers, then the rest
  int order[CKV_CSA2_MAX_LAYERS], n_first = 0, n = 0;
  for (int l = 0; l < L && n_first < kLayersPerLaunch; ++l)
    if (g->role[root[l]] == CKV_CSA2_FULL) order[n++] = l, ++n_first;
  for (int l = 0; l < L; ++l) {
    bool placed = false;
    for (int j = 0; j < n_first; ++j) placed |= order[j] == l;
    if (!placed) order[n++] = l;
  }
  AttnArgs la[CKV_CSA2_MAX_LAYERS];
  for (int j0 = 0, gi = 0; j0 < L; ++gi) {
    // the first launch: the Full-derived layers; then the rest, evenly
    int n_g;
    if (gi == 0 && n_first > 0) {
      n_g = n_first;
    } else {
      const int left = L - j0, n_launch = (left + kLayersPerLaunch - 1) / kLayersPerLaunch;
      n_g = left / n_launch;
    }
    // the first launch on the side stream, beside the Reindex passes; the
    // later ones after those passes on the caller's stream
    const cudaStream_t ls = gi == 0 ? side->s : st;
    int rows_max = 0;
    for (int j = j0; j < j0 + n_g; ++j) {
      const int r = topk + (int)g->win[g->kv_src[order[j]]].cap;
      rows_max = rows_max > r ? rows_max : r;
    }
    const PairChoice pc = choose_pairs(B * n_g, rows_max);
    for (int j = j0; j < j0 + n_g; ++j) {
      const int l = order[j], k = g->kv_src[l];
      la[j] = attn_args(&g->kv[k], &g->win[k], win_len, g->q[l], H, sm_scale, g->out[l], g->lse[l], dst);
      set_rope(la[j], &g->rope);   // checked before any launch
      la[j].idx = own[root[l]];
      la[j].topk = topk;
      la[j].G = pc.G;
      la[j].cluster_all = pc.cluster_all;
      attn_set_ws(la[j], attn_region, B, CKV_CSA2_MAX_LAYERS, j0);
      if (g->role[l] == CKV_CSA2_REUSE && g->idx_out[l]) {
        s = cuda_status(cudaMemcpyAsync(g->idx_out[l], own[root[l]], (size_t)B * topk * 4,
                                        cudaMemcpyDeviceToDevice, ls));
        if (s) return s;
      }
    }
    s = cuda_status(launch_attention_layers(la + j0, n_g, B, ls));
    if (s) return s;
    j0 += n_g;
  }
  // everything on the side stream is done before the caller's stream goes on
  s = cuda_status(cudaEventRecord(side->re, side->s));
  if (s) return s;
  return cuda_status(cudaStreamWaitEvent(st, side->re, 0));
}

ckv_status ckv_csa2_group_decode(const ckv_csa2_group* g, const int32_t* n_comp,
                                 int32_t n_comp_max, const int32_t* win_len, int32_t B,
                                 int32_t H, int32_t HI, int32_t topk, float sm_scale,
                                 const ckv_plane* append_dst, const void* append_src_bf16,
                                 const int64_t* append_slot, int32_t n_append, void* ws,
                                 size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("ckv_csa2_group_decode");
  if (!g || g->n_layers < 1 || g->n_layers > CKV_CSA2_MAX_LAYERS) return CKV_ERR_INVALID;
  const int L = g->n_layers;
  if (g->role[0] != CKV_CSA2_FULL) return CKV_ERR_INVALID;
  const int pool_len = g->pool_len;
  if (pool_len < topk || pool_len > kMaxPool) return CKV_ERR_INVALID;
  bool any_reindex = false;
  for (int l = 0; l < L; ++l) {
    const int r = g->role[l];
    if (r < CKV_CSA2_FULL || r > CKV_CSA2_REUSE) return CKV_ERR_INVALID;
    if (r == CKV_CSA2_REUSE && (g->idx_src[l] < 0 || g->idx_src[l] >= l)) return CKV_ERR_INVALID;
    if (g->kv_src[l] < 0 || g->kv_src[l] >= L) return CKV_ERR_INVALID;
    if (r != CKV_CSA2_REUSE) {
      ckv_status s = check_index_args(&g->idx_keys, n_comp, B, n_comp_max, g->q_idx[l], g->w[l],
                                      HI, topk, nullptr, 0, reinterpret_cast<int32_t*>(1),
                                      r == CKV_CSA2_FULL ? reinterpret_cast<int32_t*>(1) : nullptr,
                                      pool_len);
      if (s) return s;
    }
    any_reindex |= r == CKV_CSA2_REINDEX;
    const int k = g->kv_src[l];
    ckv_status s = check_attn_common(&g->kv[k], &g->win[k], win_len, B, g->q[l], H, g->out[l], sm_scale);
    if (s) return s;
    if (n_comp_max > g->kv[k].cap) return CKV_ERR_INVALID;
    // the group's attention launches share one kernel instance: one cache format for all
    if (g->kv[k].fmt != g->kv[g->kv_src[0]].fmt) return CKV_ERR_UNSUPPORTED;
  }
  (void)any_reindex;
  if (topk > kMaxTopk) return CKV_ERR_UNSUPPORTED;
  if (g->rope.pos && !g->rope.inv_freq) return CKV_ERR_INVALID;
  if (n_append > 0) {
    if (!append_dst || !append_src_bf16 || !append_slot || !aligned16(append_src_bf16))
      return CKV_ERR_INVALID;
    ckv_status s = check_plane(append_dst, append_dst->dim, 1);
    if (s) return s;
  }
  const size_t need = ckv_workspace_bytes(CKV_OP_CSA2, B, H, HI, n_comp_max, topk, pool_len);
  ckv_status s = check_ws(ws, ws_bytes, need);
  if (s) return s;
  {
    // Replaying a captured group call has faulted on GB300 with no cause
    // found: refuse to be captured, before anything is enqueued.  A capture
    // in global mode on another stream makes the legacy default stream's
    // query fail with cudaErrorStreamCaptureImplicit: refused as well.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t ce = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs);
    if (ce == cudaErrorStreamCaptureImplicit) {
      (void)cudaGetLastError();
      return CKV_ERR_UNSUPPORTED;
    }
    if (ce != cudaSuccess) return cuda_status(ce);
    if (cs != cudaStreamCaptureStatusNone) return CKV_ERR_UNSUPPORTED;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  DevStatus* dst = reinterpret_cast<DevStatus*>(w8);
  const size_t full = index_ws_bytes(B, n_comp_max, false, 0);
  const size_t re = index_ws_bytes(B, n_comp_max, true, pool_len);
  uint8_t* idx_region = w8 + kStatusBytes;
  int32_t* pool_buf = reinterpret_cast<int32_t*>(idx_region + align_up(full > re ? full : re, 256));
  int32_t* idxbuf = pool_buf + align_up((size_t)B * pool_len * 4, 256) / 4;
  uint8_t* attn_region = reinterpret_cast<uint8_t*>(idxbuf) +
                         align_up((size_t)CKV_CSA2_MAX_LAYERS * B * topk * 4, 256);

  if (n_append > 0) {
    s = cuda_status(launch_append(*append_dst, append_src_bf16, append_slot, n_append, dst, st));
    if (s) return s;
  }
  // Layers whose indices come from a Reindex pass (directly or by reuse)
  // wait for it; the others need only the Full pass of layer 0.  With one
  // Full layer and at least one Reindex layer, the first attention launch
  // (Full-derived layers only) runs on a side stream beside the Reindex
  // passes on the caller's stream.
  {
    int root[CKV_CSA2_MAX_LAYERS];
    bool one_full = true, any_re = false;
    for (int l = 0; l < L; ++l) {
      root[l] = g->role[l] == CKV_CSA2_REUSE ? root[g->idx_src[l]] : l;
      if (l > 0 && g->role[l] == CKV_CSA2_FULL) one_full = false;
      any_re |= g->role[l] == CKV_CSA2_REINDEX;
    }
    if (one_full && any_re && L >= 2)
      return csa2_group_overlapped(g, root, n_comp, n_comp_max, win_len, B, H, HI, topk, sm_scale,
                                   pool_len, idxbuf, pool_buf, idx_region, attn_region, dst, st);
  }
  const int32_t* layer_idx[CKV_CSA2_MAX_LAYERS];
  for (int l = 0; l < L; ++l) {
    int32_t* own = g->idx_out[l] ? g->idx_out[l] : idxbuf + (size_t)l * B * topk;
    if (g->role[l] == CKV_CSA2_FULL) {
      s = run_index(&g->idx_keys, n_comp, B, n_comp_max, g->q_idx[l], g->w[l], HI, topk, nullptr,
                    0, own, pool_buf, pool_len, nullptr, dst, idx_region, st);
      layer_idx[l] = own;
    } else if (g->role[l] == CKV_CSA2_REINDEX) {
      s = run_index(&g->idx_keys, n_comp, B, n_comp_max, g->q_idx[l], g->w[l], HI, topk, pool_buf,
                    pool_len, own, nullptr, 0, nullptr, dst, idx_region, st);
      layer_idx[l] = own;
    } else {
      layer_idx[l] = layer_idx[g->idx_src[l]];
      if (g->idx_out[l])
        s = cuda_status(cudaMemcpyAsync(g->idx_out[l], layer_idx[l], (size_t)B * topk * 4,
                                        cudaMemcpyDeviceToDevice, st));
    }
    if (s) return s;
  }
  // the layers' attention in as few launches as the parameter block allows
  // (grid z = layer within a launch), split evenly: 6 layers -> 3 + 3
  AttnArgs la[CKV_CSA2_MAX_LAYERS];
  const int n_launch = (L + kLayersPerLaunch - 1) / kLayersPerLaunch;
  for (int gi = 0, l0 = 0; gi < n_launch; ++gi) {
    const int n_g = (L - l0) / (n_launch - gi);
    // one shape per launch: its tightest layer decides
    int rows_max = 0;
    for (int l = l0; l < l0 + n_g; ++l) {
      const int r = topk + (int)g->win[g->kv_src[l]].cap;
      rows_max = rows_max > r ? rows_max : r;
    }
    const PairChoice pc = choose_pairs(B * n_g, rows_max);
    for (int l = l0; l < l0 + n_g; ++l) {
      const int k = g->kv_src[l];
      la[l] = attn_args(&g->kv[k], &g->win[k], win_len, g->q[l], H, sm_scale, g->out[l], g->lse[l], dst);
      set_rope(la[l], &g->rope);   // checked before any launch
      la[l].idx = layer_idx[l];
      la[l].topk = topk;
      la[l].G = pc.G;
      la[l].cluster_all = pc.cluster_all;
      attn_set_ws(la[l], attn_region, B, CKV_CSA2_MAX_LAYERS, l0);
    }
    s = cuda_status(launch_attention_layers(la + l0, n_g, B, st));
    if (s) return s;
    l0 += n_g;
  }
  return CKV_OK;
}

ckv_status ckv_debug_wait_probe(void* ws, size_t ws_bytes, int32_t mode, uint32_t limit_us,
                                void* stream) {
  NvtxRange nvtx_range("ckv_debug_wait_probe");
  if (mode != 0 && mode != 1) return CKV_ERR_INVALID;
  if (limit_us < 1 || limit_us > 2000000u) return CKV_ERR_INVALID;
  // mode 1 spins on the first word after the status block, which the
  // caller keeps zero
  ckv_status s = check_ws(ws, ws_bytes, kStatusBytes + (mode == 1 ? 256 : 0));
  if (s) return s;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<DevStatus*>(w8), reinterpret_cast<const uint32_t*>(w8 + kStatusBytes), mode,
      (uint64_t)limit_us * 1000ull);
  return cuda_status(cudaGetLastError());
}

ckv_status ckv_read_device_status(void* ws, void* stream) {
  if (!ws) return CKV_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  int32_t code = 0;
  if (cudaMemcpy(&code, ws, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CKV_ERR_CUDA;
  if (code != 0) {
    if (cudaMemset(ws, 0, kStatusBytes) != cudaSuccess) return CKV_ERR_CUDA;
  }
  return code;
}

const char* ckv_status_string(ckv_status s) {
  switch (s) {
    case CKV_OK: return "CKV_OK";
    case CKV_ERR_INVALID: return "CKV_ERR_INVALID";
    case CKV_ERR_UNSUPPORTED: return "CKV_ERR_UNSUPPORTED";
    case CKV_ERR_CUDA: return "CKV_ERR_CUDA";
    case CKV_ERR_WORKSPACE: return "CKV_ERR_WORKSPACE";
    case CKV_ERR_TIMEOUT: return "CKV_ERR_TIMEOUT";
    case CKV_ERR_DEVICE_BOUNDS: return "CKV_ERR_DEVICE_BOUNDS";
    default: return "CKV_ERR_UNKNOWN";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Static-scratch variant of csa_index_topk (no allocation by anyone).  The
// scratch is this file's device array; host code finds its device address
// with cudaGetSymbolAddress once per device (the array's name is only a
// host-side stand-in) and passes that address to the same kernels.
static __device__ __align__(256) uint8_t g_index_scratch[CKV_STATIC_SCRATCH_BYTES];
static void* g_index_scratch_dev[kOnceDevices] = {};

// Device address of the static scratch on the current device, looked up
// once per device with that device current.
static cudaError_t static_scratch(uint8_t** out) {
  static DeviceOnce once;
  const cudaError_t e = once_per_device(once, [](int d) {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_index_scratch);
    g_index_scratch_dev[d] = p;
    return r != cudaSuccess ? r : p == nullptr ? cudaErrorUnknown : cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  int dev = -1;
  const cudaError_t g = cudaGetDevice(&dev);
  if (g != cudaSuccess) return g;
  *out = static_cast<uint8_t*>(g_index_scratch_dev[dev]);
  return cudaSuccess;
}

extern "C" ckv_status ckv_csa_index_topk_static(const ckv_plane* idx_keys, const int32_t* n_comp,
                                                int32_t B, int32_t n_comp_max,
                                                const void* q_idx_bf16, const float* w,
                                                int32_t HI, int32_t topk, const int32_t* pool,
                                                int32_t pool_len, int32_t* out_idx,
                                                int32_t* out_pool, int32_t pool_out,
                                                float* dbg_scores, void* stream) {
  NvtxRange nvtx_range("ckv_csa_index_topk_static");
  ckv_status s = check_index_args(idx_keys, n_comp, B, n_comp_max, q_idx_bf16, w, HI, topk, pool,
                                  pool_len, out_idx, out_pool, pool_out);
  if (s) return s;
  const bool pool_mode = pool != nullptr;
  const IndexLayout L = index_layout(B, n_comp_max, pool_mode, pool_mode ? pool_len : 0);
  if (kStatusBytes + L.bytes > (size_t)CKV_STATIC_SCRATCH_BYTES) return CKV_ERR_WORKSPACE;
  uint8_t* w8 = nullptr;
  s = cuda_status(static_scratch(&w8));
  if (s) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The per-sequence tickets and histograms must start at zero (a call
  // that ran with other sizes may have left its own layout's state behind).
  // The status word is not cleared: it is sticky until
  // ckv_read_static_status reads it.
  s = cuda_status(cudaMemsetAsync(w8 + kStatusBytes, 0, index_zero_bytes(B), st));
  if (s) return s;
  return run_index(idx_keys, n_comp, B, n_comp_max, q_idx_bf16, w, HI, topk, pool, pool_len,
                   out_idx, out_pool, pool_out, dbg_scores, reinterpret_cast<DevStatus*>(w8),
                   w8 + kStatusBytes, st);
}

extern "C" ckv_status ckv_read_static_status(void* stream) {
  NvtxRange nvtx_range("ckv_read_static_status");
  uint8_t* w8 = nullptr;
  ckv_status s = cuda_status(static_scratch(&w8));
  if (s) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  int32_t code = 0;
  if (cudaMemcpy(&code, w8, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess) return CKV_ERR_CUDA;
  if (code != 0 && cudaMemset(w8, 0, kStatusBytes) != cudaSuccess) return CKV_ERR_CUDA;
  return code;
}

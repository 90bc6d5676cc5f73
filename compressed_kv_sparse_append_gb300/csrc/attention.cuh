// Shared declarations of the attention kernels.
#pragma once

#include <cuda.h>   // CUtensorMap (the driver entry point is fetched at run time)

#include "common.cuh"

namespace ckv {

constexpr int kMaxTopk = 2048;    // selected rows held per sequence
constexpr int kMaxHeads = 128;    // query heads (one 128-row MMA tile)
// One CTA's partial, in 4-byte words: O / l as fp16 [32 chunks of 8 columns]
// [128 heads] (16 bytes each), then (m, l) as f32 pairs [128].
constexpr int64_t kPartFloats = 32 * 128 * 4 + 128 * 2;

struct AttnArgs {
  const uint8_t* kv_data;
  const void* kv_scale;
  int64_t kv_cap;
  int64_t kv_rows;          // rows of the main-KV arrays (dense: B * cap)
  const int32_t* kv_bt;     // paged main KV: block table [B][kv_bt_cols], else null
  int kv_page, kv_bt_cols;
  const uint8_t* win_data;
  const void* win_scale;
  int64_t win_cap;
  int fmt, nope_block;
  const int32_t* idx;     // CSA: [B][topk] selected entries; null for HCA
  int topk;
  const int32_t* n_comp;  // HCA: [B]
  int n_comp_max;
  const int32_t* win_len; // [B]
  const __nv_bfloat16* q; // [B][H][512]
  int H;
  float scale_log2;       // sm_scale * log2(e)
  __nv_bfloat16* out;     // [B][H][512]
  float* lse;             // [B][H] or null
  int G;                  // CTA pairs per sequence
  int cluster_all;        // 1: one cluster of 2G CTAs per sequence; 0: one per pair
  float* part;            // workspace: [layer][B][2G][kPartFloats] partial O / l, m, l
  uint32_t* tickets;      // workspace: [layer][B][2] finished-CTA counters (start at 0)
  int use_tma;            // set by the launcher: contiguous BF16 rows via TMA
  int progress;           // debugging: count pipeline events in the status block
  int tag;                // set by the launcher: kArgsTag ^ layer (checked on entry)
  const int32_t* rope_pos;  // RoPE at the attention's ends: [B] query position i, or null
  const float* rope_freq;   // [32] angle per position of rope pair k
  int rope_q, rope_out;     // turn the query by +i / the output by -i
  DevStatus* st;
  CUtensorMap gmap[4];    // set by the launcher for BF16 rows: row-gather maps (main, window)
};

constexpr int kMaxPairs = 8;      // CTA pairs per sequence
// Layers per launch: the kernel's whole parameter block (two tensor maps and
// the batch) stays within 4 KB, the classic kernel-parameter limit; more
// layers take more launches.
constexpr int kLayersPerLaunch = 4;
constexpr int kArgsTag = 0x434B5641;
struct AttnBatch {
  AttnArgs layer[kLayersPerLaunch];  // one launch runs these layers (grid z = layer)
};
static_assert(2 * sizeof(CUtensorMap) + sizeof(AttnBatch) <= 4096,
              "attention parameter block above 4 KB");

cudaError_t launch_attention(const AttnArgs& a, int B, cudaStream_t stream);
int attn_max_active_clusters(int cluster_size);
// All `n` (<= kLayersPerLaunch) layers share B, G and the row format; layer
// l uses grid z = l.
cudaError_t launch_attention_layers(const AttnArgs* layers, int n, int B, cudaStream_t stream);

}  // namespace ckv

// Shared declarations of the indexer / top-k kernels.
#pragma once

#include "common.cuh"

namespace ckv {

constexpr int kIdxDim = 128;      // indexer head dim ("DeepSeek-V4 KV Cache 深度分析", §一)
constexpr int kMaxHI = 64;        // indexer heads supported
constexpr int kMaxChunk = 8192;   // entries scored per CTA
constexpr int kMaxPool = 2048;    // largest pool / top-k kept by the merge
// Key histograms: the top kBinBits bits of the order-preserving key (for
// positive scores: the exponent and 4 mantissa bits, bins of 1/16 octave).
constexpr int kBinBits = 13;
constexpr int kBinShift = 32 - kBinBits;
constexpr int kBins = 1 << kBinBits;
constexpr int kMaxChunksPerSeq = 1024;
constexpr int kSeqWords = 4;      // per sequence: ticket, top bin + 1, kBins - low bin, spare

struct IndexArgs {
  const uint8_t* kdata;           // indexer-key plane data
  const uint8_t* kscale;          // FP4: E4M3 scale bytes
  int64_t cap;
  const int32_t* bt;              // paged key plane: block table [B][bt_cols], else null
  int page, bt_cols;
  int64_t rows;                   // rows of the key arrays
  int fmt;                        // CKV_FMT_FP4, _FP4H or _BF16
  const int32_t* n_comp;
  int B, n_comp_max;
  const __nv_bfloat16* q_idx;
  const float* w;
  int HI;
  const int32_t* pool;            // Reindex: candidate entries, or null
  int pool_len;
  int topk, pool_out;
  int chunk, n_chunks;
  uint32_t* cand_key;             // workspace [B][n_chunks][chunk] candidate keys
  int32_t* cand_idx;              // workspace [B][n_chunks][chunk] their entries
  uint32_t* ccount;               // workspace [B][n_chunks][2]: candidates, real keys
  uint32_t* seq_state;            // workspace [B][4]: ticket, bin range; zero between calls
  uint32_t* ghist;                // workspace [B][8192] key histogram, zero between calls
  int32_t* out_idx;
  int32_t* out_pool;
  float* dbg;
  DevStatus* st;
  int trace;                      // debugging: timeline in the status block
};

size_t index_smem_bytes();
cudaError_t launch_index_simt(const IndexArgs& a, cudaStream_t stream);
bool index_umma_supported(const IndexArgs& a, int64_t batch_rows);
cudaError_t launch_index_umma(const IndexArgs& a, int64_t batch_rows, cudaStream_t stream);

}  // namespace ckv

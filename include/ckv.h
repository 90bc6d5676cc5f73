/*
 * ckv.h -- C ABI of libckv: decode-time attention over the compressed KV
 * caches of DeepSeek-V4 (CSA / HCA) and V4.1-Flash (CSA2, FP4 main KV), for
 * GB300 (sm_103a).
 *
 * Sources (page title, section):
 *   [KVC]  "DeepSeek-V4 KV Cache 深度分析": §二 entry layout (512-d latent whose
 *          last 64 dims carry RoPE; nope in FP8, rope in BF16), §三 CSA/HCA
 *          (ratio 4 with top-k, ratio 128 dense, 128-token window), §四 indexer
 *          (128-d FP4 keys, top-k), §六 precision, §十一 flow chart.
 *   [V41]  "DeepSeek, KV 캐시를 토큰당 890바이트로 줄인 V4.1-Flash 공개",
 *          핵심 내용: CSA2 Full / Reindex / Reuse, FP4 E2M1 with one E4M3
 *          scale per 16 channels.
 *   [890]  "KV cache 890 bajtów na token", "Trzy mechanizmy": shared main KV
 *          and indexer key across layers, indexer pool of the Full layer.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless marked [host].  The caller owns
 *     every buffer; the library allocates no device memory and keeps no
 *     state between calls (apart from the per-device launch attributes it
 *     sets once, and the side stream and two events that
 *     ckv_csa2_group_decode creates on its first call in each host thread
 *     and device).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and return after enqueueing.  The
 *     kernels are launched with programmatic stream serialisation: one may
 *     begin launching while the previous work in the stream finishes, but it
 *     touches no global memory (inputs, outputs, workspace) before that work
 *     is complete, so stream order holds as usual.
 *   - Arguments are validated on the host first.  A host-detected error
 *     returns CKV_ERR_INVALID / CKV_ERR_UNSUPPORTED / CKV_ERR_WORKSPACE and
 *     enqueues nothing.  A failed launch returns CKV_ERR_CUDA.
 *   - `ws` is a caller-owned device workspace of at least
 *     ckv_workspace_bytes(op, ...) bytes, 256-byte aligned, ZERO-FILLED
 *     before its first use; every call leaves it reusable (its counters
 *     return to zero).  Its first 256 bytes hold a sticky device status
 *     word: kernels that detect an out-of-range index or a bounded wait that
 *     expired record CKV_ERR_DEVICE_BOUNDS / CKV_ERR_TIMEOUT there, skip the
 *     offending access and never trap.  ckv_read_device_status() returns
 *     and clears it.  Calls that overlap on the GPU must use distinct
 *     workspaces.  Host-side, the library is thread-safe and reentrant on
 *     distinct workspaces.  On the GPU no kernel waits for CTAs outside its
 *     own thread-block cluster: where a sequence's attention spans several
 *     clusters, the last of its CTAs to finish merges their partials (a
 *     counter in the workspace), so concurrent launches from several streams
 *     cannot starve one another.  One workspace may serve, one after another, the
 *     ckv_csa_index_topk, ckv_csa_sparse_attn and ckv_hca_attn calls of a
 *     step that share the batch size B (size it for the largest): the state
 *     each keeps between calls (merge tickets, key histograms, merge
 *     counters) sits at fixed offsets after the status word, and every
 *     call's scratch lies beyond all of it.  ckv_csa2_group_decode lays out
 *     its workspace its own way: give it one of its own.
 *   - Dimensions are fixed by the pages: main-KV entries are D = 512 with
 *     R = 64 RoPE dims, indexer keys are 128-d, heads H <= 128.
 */
#ifndef CKV_H
#define CKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ckv_status;
#define CKV_OK                 0
#define CKV_ERR_INVALID       -1  /* bad argument (null, misaligned, out of range) */
#define CKV_ERR_UNSUPPORTED   -2  /* valid but not implemented shape / format      */
#define CKV_ERR_CUDA          -3  /* CUDA runtime or launch failure                */
#define CKV_ERR_WORKSPACE     -4  /* workspace missing or smaller than required    */
#define CKV_ERR_TIMEOUT       -5  /* device: a bounded wait expired                */
#define CKV_ERR_DEVICE_BOUNDS -6  /* device: an index or slot was out of range     */

/* Storage formats of a cache plane.
 *  CKV_FMT_BF16  : entry = dim x bf16 (1024 B for D = 512, 256 B for 128).
 *  CKV_FMT_MIXED : D = 512 only. Entry = 448 x E4M3 nope codes followed by
 *                  64 x bf16 rope values = 576 B ([KVC] §二, §六).  One f32
 *                  scale per block of `nope_block` nope channels in `scale`:
 *                  value = decode(code) * scale.
 *  CKV_FMT_FP4   : entry = dim/2 bytes of packed E2M1 codes, channel 2t in the
 *                  low nibble of byte t, channel 2t+1 in the high nibble; one
 *                  E4M3 scale byte per 16 channels in `scale` ([V41]).
 *  CKV_FMT_FP4H  : indexer keys only (dim 128).  The FP4 layout above, of the
 *                  Hadamard-rotated vector ([KVC] §四: Hadamard rotation, then
 *                  FP4 over all 128 dims): x H with H the Sylvester Hadamard
 *                  matrix of order 128 over sqrt(128), computed as f32
 *                  butterflies (stage h = 1, 2, ..., 64: pair (j, j + h) ->
 *                  (a + b, a - b)) and one f32 multiplication by
 *                  fl32(1/sqrt(128)).  Scoring against such keys rotates the
 *                  query the same way before quantising it; an orthogonal
 *                  rotation of both sides leaves q . k unchanged. */
#define CKV_FMT_BF16  0
#define CKV_FMT_MIXED 1
#define CKV_FMT_FP4   2
#define CKV_FMT_FP4H  3

/* One cache plane (main KV, window ring, or indexer keys) of `batch`
 * sequences with `cap` entry slots each.  The plane struct itself is [host].
 *
 * Dense (block_table == NULL): entry (b, pos) is row b * cap + pos: it lives
 * at data + row * entry_bytes, its scales at scale + row * n_scales *
 * scale_size.
 *
 * Paged (block_table != NULL): the rows of the plane are n_pages pages of
 * page_size rows each; sequence b's logical block j (positions
 * [j * page_size, (j + 1) * page_size)) is page block_table[b * (cap /
 * page_size) + j], so entry (b, pos) is row
 *   block_table[b * (cap / page_size) + pos / page_size] * page_size
 *     + pos % page_size,
 * addressed as above.  page_size is a multiple of 128 and divides cap;
 * every page id is in [0, n_pages).  The pages define no layout of their own
 * (they allocate the cache dense, [batch][cap][entry]); paging lets a
 * serving engine grow and share sequences' caches in pages.  Main-KV and
 * indexer-key planes may be paged; window planes are dense.
 * data and scale are 16-byte aligned. */
typedef struct ckv_plane {
  int32_t fmt;        /* CKV_FMT_*                                           */
  int32_t dim;        /* 512 (main KV, window) or 128 (indexer keys)         */
  int32_t nope_block; /* CKV_FMT_MIXED: 448 (one scale per entry) or 64      */
  int32_t batch;      /* sequences                                           */
  int64_t cap;        /* entry slots (logical positions) per sequence        */
  void   *data;       /* [rows][entry_bytes]; rows = batch * cap (dense) or
                         n_pages * page_size (paged)                         */
  void   *scale;      /* MIXED: f32 [rows][448/nope_block];
                         FP4 / FP4H: u8 [rows][dim/16] (E4M3 codes);
                         BF16:  NULL                                         */
  const int32_t *block_table; /* NULL (dense) or [batch][cap / page_size]    */
  int32_t page_size;  /* paged: rows per page (multiple of 128)              */
  int32_t n_pages;    /* paged: pages in data / scale                        */
} ckv_plane;

/* Workspace sizing.  `op` is one of CKV_OP_*; unused arguments may be 0.
 * The attention ops (CKV_OP_SPARSE_ATTN, CKV_OP_HCA_ATTN, and CKV_OP_CSA2
 * for each of its up to CKV_CSA2_MAX_LAYERS layers) keep one partial
 * (output normalised by its own row sum, running max and sum) per CTA of a sequence in the
 * workspace for the final merge, plus one counter per sequence, layer and
 * half that elects the CTA doing the merge: about 1.1 MB per sequence and
 * layer.  The single-op calls (CKV_OP_INDEX_TOPK, CKV_OP_SPARSE_ATTN,
 * CKV_OP_HCA_ATTN) also reserve the shared between-call state of all three
 * for B (about 16 KB per sequence; see the workspace note above). */
#define CKV_OP_APPEND      0
#define CKV_OP_INDEX_TOPK  1
#define CKV_OP_SPARSE_ATTN 2
#define CKV_OP_HCA_ATTN    3
#define CKV_OP_CSA2        4
size_t ckv_workspace_bytes(int32_t op, int32_t B, int32_t H, int32_t HI,
                           int32_t n_comp_max, int32_t topk, int32_t pool_len);

/* Append-side quantise and store ([KVC] §二 code evidence: the latent's first
 * 448 dims quantised to FP8, the 64 RoPE dims kept BF16; [V41] / [890]: FP4
 * E2M1 with one E4M3 scale per 16 channels, used for the V4.1 main KV and
 * here also for the 128-d indexer keys of [KVC] §四).
 *   dst      [host] destination plane (any format; dim 512 or 128).
 *   src_bf16 [n][dst->dim] bf16 rows, already normalised and rotated.
 *   slot     [n] int64: destination row of the plane: b * cap + pos for a
 *            dense plane, page * page_size + offset for a paged one (the
 *            caller owns the page allocation).  A negative slot skips the
 *            row; a slot beyond the plane's rows skips it and records
 *            CKV_ERR_DEVICE_BOUNDS.
 * Quantisation (bit-exact contract):
 *   MIXED: s = fl32(amax_block / 448) (f32), code_i = E4M3_rn_satfinite(
 *          fl32(x_i / s)); rope dims copied as bf16.
 *   FP4:   s = E4M3_rn_satfinite(fl32(amax16 / 6)), code_i =
 *          E2M1_rn_satfinite(fl32(x_i / decode(s))).
 *   FP4H:  the same on the Hadamard-rotated row (dim 128; see CKV_FMT_FP4H).
 *   Codes carry the sign of x (tiny negatives give the negative-zero code);
 *   a block whose scale is zero stores all-zero codes. */
ckv_status ckv_kv_append_quant(const ckv_plane *dst, const void *src_bf16,
                               const int64_t *slot, int32_t n,
                               void *ws, size_t ws_bytes, void *stream);

/* Several appends in one launch (the same passages as ckv_kv_append_quant):
 * plane k receives n[k] rows src_bf16[k] at slot[k], stored bit-exactly as
 * ckv_kv_append_quant(&dst[k], src_bf16[k], slot[k], n[k], ...) stores them.
 * A decode step appends to several planes (the main KV and the indexer
 * keys); one launch instead of one per plane shortens the step's chain of
 * dependent launches.
 *   dst      [host] n_planes plane descriptors, 1 <= n_planes <=
 *            CKV_APPEND_MAX_PLANES, with distinct data arrays.
 *   src_bf16 [host] n_planes device pointers, each [n[k]][dst[k].dim] bf16.
 *   slot     [host] n_planes device pointers, each [n[k]] int64 (as above).
 *   n        [host] n_planes row counts (>= 0).
 * Validation, workspace and device status as ckv_kv_append_quant. */
#define CKV_APPEND_MAX_PLANES 4
ckv_status ckv_kv_append_quant_multi(const ckv_plane *dst, const void *const *src_bf16,
                                     const int64_t *const *slot, const int32_t *n,
                                     int32_t n_planes, void *ws, size_t ws_bytes, void *stream);

/* Lightning-indexer score + exact top-k ([KVC] §四; score definition
 * s_j = sum_h w_h * ReLU(q_h . k_j) on the dequantised values; for FP4 keys
 * the query is first quantised with the same E2M1 + E4M3/16 block
 * quantiser, "computed entirely in FP4").
 *   idx_keys   [host] indexer-key plane, dim 128, CKV_FMT_FP4, _FP4H or _BF16.
 *   n_comp     [B] int32: valid entries of each sequence (<= n_comp_max).
 *   n_comp_max [host] upper bound of n_comp (sizes the grid).
 *   q_idx_bf16 [B][HI][128] bf16 indexer queries; w [B][HI] f32 weights.
 *   topk       entries to select (1..2048).
 *   pool       NULL: score every entry [0, n_comp[b]).  Otherwise
 *              [B][pool_len] int32 candidate entries (-1 = unused); only
 *              those are scored (the CSA2 Reindex layer, [890]).
 *   out_idx    [B][topk] int32: the top-k entries, ascending, -1 padded.
 *              Order: score descending, then index ascending (lower index
 *              wins a tie); -0.0 counts as +0.0.
 *   out_pool   NULL or [B][pool_out] int32: the top-pool_out set under the
 *              same order, ascending, -1 padded (CSA2 Full layer's pool);
 *              pool_out >= topk; requires pool == NULL.
 *   dbg_scores NULL or [B][n_comp_max] f32: every computed score at its
 *              entry index (diagnostics; costs bandwidth).
 * Scores are f32 with an accumulation order the tensor cores fix; the
 * selection is exact on those f32 scores. */
ckv_status ckv_csa_index_topk(const ckv_plane *idx_keys, const int32_t *n_comp,
                              int32_t B, int32_t n_comp_max,
                              const void *q_idx_bf16, const float *w, int32_t HI,
                              int32_t topk, const int32_t *pool, int32_t pool_len,
                              int32_t *out_idx, int32_t *out_pool, int32_t pool_out,
                              float *dbg_scores, void *ws, size_t ws_bytes,
                              void *stream);

/* csa_index_topk for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment convenience.  Some callers cannot
 * call cudaMalloc at all -- plug-ins of serving engines that own every device
 * allocation, or embedded runtimes whose memory plan is fixed before they
 * start -- and so cannot provide the workspace of ckv_csa_index_topk.  This
 * entry point computes exactly the same outputs with its scratch in a
 * statically sized device array inside libckv (CKV_STATIC_SCRATCH_BYTES, held
 * on every GPU that loads the library until the process exits); it calls no
 * allocating routine.
 *   Arguments as ckv_csa_index_topk, without ws / ws_bytes.
 *   Returns CKV_ERR_WORKSPACE when the call needs more scratch than
 *   CKV_STATIC_SCRATCH_BYTES (see ckv_workspace_bytes(CKV_OP_INDEX_TOPK, ...)).
 *   The first call on a device looks the array up (cudaGetSymbolAddress)
 *   with that device current.  Every call first clears the scratch's
 *   counters on `stream`.
 *   All calls share the one array, which keeps the last call's contents:
 *   calls that overlap on the GPU (different streams) race and must be
 *   serialised by the caller.  Device-side range errors (a pool entry at or
 *   beyond n_comp) are recorded in the array's own sticky status word; read
 *   it with ckv_read_static_status. */
#define CKV_STATIC_SCRATCH_BYTES (8u << 20)
ckv_status ckv_csa_index_topk_static(const ckv_plane *idx_keys, const int32_t *n_comp,
                                     int32_t B, int32_t n_comp_max,
                                     const void *q_idx_bf16, const float *w, int32_t HI,
                                     int32_t topk, const int32_t *pool, int32_t pool_len,
                                     int32_t *out_idx, int32_t *out_pool, int32_t pool_out,
                                     float *dbg_scores, void *stream);

/* Synchronises `stream`, returns the sticky device status of the static
 * scratch of ckv_csa_index_topk_static on the current device (CKV_OK,
 * CKV_ERR_DEVICE_BOUNDS or CKV_ERR_TIMEOUT) and clears it.  The pages have no
 * counterpart. */
ckv_status ckv_read_static_status(void *stream);

/* CSA sparse attention ([KVC] §十一 flow chart: attention over the selected
 * entries followed by the sliding window; §五: each entry is both key and
 * value).  One softmax over the union of the selected rows and the valid
 * window rows:  o_h = sum_j softmax_j(sm_scale * q_h . e_j) e_j,
 * lse_h = log sum_j exp(sm_scale * q_h . e_j).
 *   kv, win  [host] main-KV and window planes of the same format (dim 512).
 *   win_len  [B] int32: valid window slots [0, win_len[b]) (<= win->cap).
 *   idx      [B][topk] int32 entries of kv (-1 = none; >= kv->cap is skipped
 *            and records CKV_ERR_DEVICE_BOUNDS).  The call has no n_comp: an
 *            entry below kv->cap is attended as whatever its slot holds, so
 *            callers pass entries that have been written (the output of
 *            ckv_csa_index_topk only names entries below its n_comp).
 *   q_bf16   [B][H][512] bf16, H <= 128.
 *   out_bf16 [B][H][512] bf16; lse NULL or [B][H] f32 (natural log; -inf when
 *            there is no row to attend, with o = 0). */
ckv_status ckv_csa_sparse_attn(const ckv_plane *kv, const ckv_plane *win,
                               const int32_t *win_len, const int32_t *idx,
                               int32_t B, int32_t topk, const void *q_bf16,
                               int32_t H, float sm_scale, void *out_bf16,
                               float *lse, void *ws, size_t ws_bytes, void *stream);

/* RoPE at the two ends of the attention ([KVC] §五, three RoPE sites: the
 * query, each compressed entry, and the core attention output at position
 * -i).  Entries reach the cache already rotated; these two sites are part of
 * the attention step.  The last 64 latent dims form 32 pairs of adjacent dims
 * (448 + 2k, 449 + 2k), each a complex number (real part first); pair k
 * turns by the angle pos * inv_freq[k].
 *   pos        [B] int32: position i of each sequence's query token.
 *   inv_freq   [32] f32: angle per position of pair k (the model's frequency
 *              table, e.g. 10000^(-2k/64), scaled or not).
 *   rotate_q   nonzero: the query's last 64 dims turn by +i before the
 *              products (the rotated query is rounded to bf16).
 *   rotate_out nonzero: the output's last 64 dims turn by -i before the
 *              output is rounded to bf16 (the lse does not change).
 * The angle is reduced modulo 2 pi in double precision, then its sine and
 * cosine are taken in f32 (absolute error about 2^-21).  The struct itself
 * is [host]. */
typedef struct ckv_rope {
  const int32_t *pos;
  const float   *inv_freq;
  int32_t        rotate_q;
  int32_t        rotate_out;
} ckv_rope;

/* ckv_csa_sparse_attn with RoPE at the query and / or the output (rope
 * [host], NULL = none; see ckv_rope). */
ckv_status ckv_csa_sparse_attn_rope(const ckv_plane *kv, const ckv_plane *win,
                                    const int32_t *win_len, const int32_t *idx,
                                    int32_t B, int32_t topk, const void *q_bf16,
                                    int32_t H, float sm_scale, void *out_bf16,
                                    float *lse, const ckv_rope *rope, void *ws,
                                    size_t ws_bytes, void *stream);

/* HCA dense attention ([KVC] §三: ratio-128 entries, no sparse selection,
 * dense attention over all entries plus the 128-token window).  Same
 * formula as ckv_csa_sparse_attn over entries [0, n_comp[b]) and the window.
 *   n_comp [B] int32 (<= n_comp_max <= kv->cap). */
ckv_status ckv_hca_attn(const ckv_plane *kv, const int32_t *n_comp,
                        int32_t n_comp_max, const ckv_plane *win,
                        const int32_t *win_len, int32_t B, const void *q_bf16,
                        int32_t H, float sm_scale, void *out_bf16, float *lse,
                        void *ws, size_t ws_bytes, void *stream);

/* ckv_hca_attn with RoPE at the query and / or the output (rope [host],
 * NULL = none; see ckv_rope). */
ckv_status ckv_hca_attn_rope(const ckv_plane *kv, const int32_t *n_comp,
                             int32_t n_comp_max, const ckv_plane *win,
                             const int32_t *win_len, int32_t B, const void *q_bf16,
                             int32_t H, float sm_scale, void *out_bf16, float *lse,
                             const ckv_rope *rope, void *ws, size_t ws_bytes,
                             void *stream);

/* CSA2 group decode ([V41] 핵심 내용; [890] "Trzy mechanizmy").  Layer roles:
 *   FULL    scores every entry of `idx_keys` with its own q_idx / w, keeps
 *           the top-pool_len pool and the top-k;
 *   REINDEX rescoring of the most recent FULL layer's pool with its own
 *           q_idx / w against the same indexer keys; takes the pool's top-k;
 *   REUSE   takes the indices of layer idx_src[l] unchanged.
 * Every layer then attends (as ckv_csa_sparse_attn) to the main KV and
 * window of layer kv_src[l].  Before the layers run, the call appends
 * n_append rows to `append_dst` (as ckv_kv_append_quant).  The layers'
 * attention runs in launches of at most four layers each, so that every
 * launch's parameter block stays within the classic 4 KB.  With one FULL
 * layer (layer 0) and at least one REINDEX layer, the first attention
 * launch -- up to four layers whose indices come from the FULL pass -- runs
 * on a side stream of the library's own (one per host thread and device,
 * made on first use) beside the REINDEX passes, which run on `stream`
 * followed there by the attention of the remaining layers; `stream` finally
 * waits for the side stream, so everything the call enqueues is ordered
 * before the next work on `stream` (six layers FULL, REINDEX, 4 x REUSE of
 * layer 0: launches of four and two).  Otherwise the passes run in layer order on
 * `stream` (six layers: two launches of three).  The call refuses
 * to be captured into a CUDA graph: on
 * a capturing stream it returns CKV_ERR_UNSUPPORTED and enqueues nothing
 * (replaying a captured group call faulted on GB300, cause not found; eager
 * calls are not affected). */
#define CKV_CSA2_FULL    0
#define CKV_CSA2_REINDEX 1
#define CKV_CSA2_REUSE   2
#define CKV_CSA2_MAX_LAYERS 8
typedef struct ckv_csa2_group {
  int32_t n_layers;                       /* 1..8 (6 in V4.1-Flash)            */
  int32_t role[CKV_CSA2_MAX_LAYERS];      /* CKV_CSA2_*; layer 0 must be FULL  */
  int32_t kv_src[CKV_CSA2_MAX_LAYERS];    /* layer whose main KV / window to use */
  int32_t idx_src[CKV_CSA2_MAX_LAYERS];   /* REUSE: earlier layer to copy from */
  ckv_plane kv[CKV_CSA2_MAX_LAYERS];      /* main KV per layer (dim 512)       */
  ckv_plane win[CKV_CSA2_MAX_LAYERS];     /* window per layer                  */
  ckv_plane idx_keys;                     /* FULL layer's indexer keys (128-d) */
  const void  *q[CKV_CSA2_MAX_LAYERS];    /* [B][H][512] bf16                   */
  const void  *q_idx[CKV_CSA2_MAX_LAYERS];/* [B][HI][128] bf16 (FULL/REINDEX)   */
  const float *w[CKV_CSA2_MAX_LAYERS];    /* [B][HI] f32 (FULL/REINDEX)         */
  void    *out[CKV_CSA2_MAX_LAYERS];      /* [B][H][512] bf16                   */
  float   *lse[CKV_CSA2_MAX_LAYERS];      /* NULL or [B][H] f32                 */
  int32_t *idx_out[CKV_CSA2_MAX_LAYERS];  /* NULL or [B][topk] int32: indices used */
  int32_t  pool_len;                      /* candidate pool of the FULL layer  */
  ckv_rope rope;                          /* RoPE of every layer's query / output
                                             (pos == NULL: none; see ckv_rope) */
} ckv_csa2_group;

ckv_status ckv_csa2_group_decode(const ckv_csa2_group *g, const int32_t *n_comp,
                                 int32_t n_comp_max, const int32_t *win_len,
                                 int32_t B, int32_t H, int32_t HI, int32_t topk,
                                 float sm_scale, const ckv_plane *append_dst,
                                 const void *append_src_bf16,
                                 const int64_t *append_slot, int32_t n_append,
                                 void *ws, size_t ws_bytes, void *stream);

/* Failure-path check of the bounded waits (the pages have no counterpart).
 * Every spin-wait in the kernels gives up after a limit (2 s), records
 * CKV_ERR_TIMEOUT in the workspace status word and lets the kernel return,
 * so that a lost arrival never hangs the GPU.  This call launches one small
 * kernel that runs the same wait code on something nothing will complete:
 *   mode 0  an mbarrier phase (as the pipelines' producer/consumer waits);
 *   mode 1  the first 32-bit word after the status block, which must be
 *           zero (as the cross-CTA merge counters); needs ws_bytes >= 512.
 * The wait gives up after limit_us (1 .. 2,000,000) microseconds; the
 * status then reads CKV_ERR_TIMEOUT (ckv_read_device_status) and the GPU
 * context stays usable.  Asynchronous on `stream`. */
ckv_status ckv_debug_wait_probe(void *ws, size_t ws_bytes, int32_t mode, uint32_t limit_us,
                                void *stream);

/* Synchronises `stream`, returns the sticky device status recorded in `ws`
 * (CKV_OK, CKV_ERR_DEVICE_BOUNDS or CKV_ERR_TIMEOUT; CKV_ERR_INVALID if an
 * attention launch found its argument block damaged and skipped the layer)
 * and clears it. */
ckv_status ckv_read_device_status(void *ws, void *stream);

/* Human-readable name of a status code (static string). */
const char *ckv_status_string(ckv_status s);

#ifdef __cplusplus
}
#endif
#endif /* CKV_H */

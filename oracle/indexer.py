"""Lightning-indexer scoring and top-k selection (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"DeepSeek-V4 KV Cache 深度分析", §四: the indexer query (128-d per indexer
head) is scored against every compressed block's indexer key and the top-k
blocks are selected; its QK activations are held and computed in FP4
(§四, quoting the paper's Section 5.2.1).  The pages give no score formula;
the workload definition used here is

    d[h, j] = q_h . k_j          (exact, float64, on dequantised values)
    s[j]    = sum_h w_h * max(d[h, j], 0)

For FP4 keys the query is quantised with the same E2M1 + E4M3/16 block
quantiser per head before the product ("computed entirely in FP4").

Top-k: the k entries with the largest score; equal scores go to the lower
index; the result is the ascending index set, padded with -1 when fewer than k
entries exist.
"""

import numpy as np

from .fp_formats import fp4_quantize, fp4_dequantize


def indexer_query(q_idx, quantize_fp4: bool, hadamard: bool = False) -> np.ndarray:
    """float64 query values as the product sees them.  With ``hadamard`` (keys
    stored Hadamard-rotated, §四) the query is rotated the same way before its
    FP4 quantisation."""
    q_idx = np.asarray(q_idx, dtype=np.float32)
    if quantize_fp4:
        if hadamard:
            from .hadamard import hadamard_rotate_f32
            q_idx = hadamard_rotate_f32(q_idx)
        packed, sc = fp4_quantize(q_idx)
        return fp4_dequantize(packed, sc)
    return q_idx.astype(np.float64)


def index_scores(q_vals, w, key_vals) -> np.ndarray:
    """s[j] = sum_h w_h * ReLU(q_h . k_j) for one sequence, float64.

    q_vals [HI, 128] and key_vals [n, 128] are the (dequantised) values."""
    q_vals = np.asarray(q_vals, dtype=np.float64)
    key_vals = np.asarray(key_vals, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    d = key_vals @ q_vals.T                      # [n, HI]
    return np.maximum(d, 0.0) @ w                # [n]


def topk_set(scores, k: int, candidates=None) -> np.ndarray:
    """Ascending indices of the top-k (ties to the lower index), -1 padded."""
    if candidates is None:
        candidates = np.arange(len(scores), dtype=np.int64)
    cand = np.asarray(candidates, dtype=np.int64)
    cand = cand[cand >= 0]
    sc = np.asarray(scores, dtype=np.float64)[cand]
    order = cand[np.lexsort((cand, -sc))]
    sel = np.sort(order[: min(k, len(order))])
    out = np.full(k, -1, dtype=np.int64)
    out[: len(sel)] = sel
    return out

"""Shared-KV decode attention over compressed entries (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"DeepSeek-V4 KV Cache 深度分析":
  * §五 (RoPE, three sites): each compressed entry serves as both key and
    value (MQA-style shared KV); the output is sum_j a_j * C_j.
  * §十一 (forward flow chart): Attention(Q, K = selected, V = selected)
    followed by the 128-token sliding window; §三: HCA attends densely to all
    ratio-128 entries plus the window, CSA to the indexer's top-k plus the
    window.

Reading: one softmax over the union of the selected rows and the valid
window rows, without de-duplication and without an attention sink.  With
tau the softmax scale (1/sqrt(512)):

    z_j = tau * q_h . e_j,   o_h = sum_j exp(z_j - m) e_j / sum_j exp(z_j - m),
    lse_h = m + log sum_j exp(z_j - m),   m = max_j z_j.

An empty row set gives o = 0 and lse = -inf.
"""

import numpy as np

from .fp_formats import dequantize_entries


def attend(q, rows, tau: float):
    """q [H, D] float, rows [n, D] float64 -> (o [H, D], lse [H]) float64."""
    q = np.asarray(q, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    H = q.shape[0]
    if rows.shape[0] == 0:
        return np.zeros_like(q), np.full(H, -np.inf)
    z = tau * (q @ rows.T)                          # [H, n]
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ rows) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def gather_rows(kv_data, kv_scale, fmt, idx, win_data, win_scale, win_len, nope_block=448):
    """float64 rows of one sequence: the entries named by ``idx`` (entries
    < 0 are padding and skipped) followed by the first ``win_len`` window
    slots."""
    idx = np.asarray(idx, dtype=np.int64)
    sel = idx[idx >= 0]
    parts = []
    if len(sel):
        parts.append(dequantize_entries(kv_data[sel], None if kv_scale is None else kv_scale[sel],
                                        fmt, nope_block))
    if win_len > 0:
        parts.append(dequantize_entries(win_data[:win_len],
                                        None if win_scale is None else win_scale[:win_len],
                                        fmt, nope_block))
    if not parts:
        return np.zeros((0, kv_data.shape[-1] if fmt != "fp4" else kv_data.shape[-1] * 2))
    return np.concatenate(parts, axis=0)


def csa_sparse_attention(q, kv_data, kv_scale, fmt, idx, win_data, win_scale, win_len, tau,
                         nope_block=448):
    """One sequence of CSA: attention over selected entries plus window."""
    rows = gather_rows(kv_data, kv_scale, fmt, idx, win_data, win_scale, win_len, nope_block)
    if rows.shape[0] == 0:
        rows = np.zeros((0, np.asarray(q).shape[-1]))
    return attend(q, rows, tau)


def hca_attention(q, kv_data, kv_scale, fmt, n_comp, win_data, win_scale, win_len, tau,
                  nope_block=448):
    """One sequence of HCA: dense attention over all n_comp entries plus
    window."""
    idx = np.arange(n_comp, dtype=np.int64)
    return csa_sparse_attention(q, kv_data, kv_scale, fmt, idx, win_data, win_scale, win_len,
                                tau, nope_block)

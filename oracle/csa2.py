"""CSA2 six-layer group decode (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"V4.1-Flash 공개", 핵심 내용 (second paragraph): layers are grouped six at a
time; the group's first layer runs in Full mode (its own KV and indexer
query, its own top-512); Reuse layers take the top-512 indices of an earlier
layer unchanged; the Reindex layer reuses the most recent KV and recomputes
only the query to re-rank.  "KV cache 890 bajtów na token", "Trzy
mechanizmy" (second mechanism): layers share the main KV and the indexer key,
and deeper layers' indexing is restricted to the candidate pool built by the
Full layer.

Readings: the Full layer's candidate pool is its top-P entries under the same
order as top-k (score descending, index ascending), P a parameter; the
Reindex layer scores only the pool entries, with its own indexer query and
head weights, against the Full layer's indexer keys, and takes its top-k;
``idx_src[l]`` names the layer whose indices a Reuse layer takes and
``kv_src[l]`` the layer whose main KV and window a layer attends to.
"""

import numpy as np

from .indexer import indexer_query, index_scores, topk_set
from .attention import csa_sparse_attention

FULL, REINDEX, REUSE = 0, 1, 2


def csa2_group_sequence(roles, kv_src, idx_src, key_vals, n_comp, q_idx, w, idx_fp4,
                        topk, pool_len, q, kv, win, win_len, tau):
    """One sequence of a CSA2 group.

    roles / kv_src / idx_src: per-layer lists.  key_vals [n, 128]: the Full
    layer's dequantised indexer keys.  q_idx[l], w[l]: indexer query and head
    weights of the Full and Reindex layers.  kv[l] = (data, scale, fmt) and
    win[l] = (data, scale) of each layer's planes.  Returns (per-layer
    indices, pool, per-layer (o, lse)).
    """
    L = len(roles)
    idx = [None] * L
    pool = None
    for l in range(L):
        if roles[l] == FULL:
            s = index_scores(indexer_query(q_idx[l], idx_fp4), w[l], key_vals[:n_comp])
            pool = topk_set(s, pool_len)
            idx[l] = topk_set(s, topk)
        elif roles[l] == REINDEX:
            assert pool is not None
            cand = pool[pool >= 0]
            s_all = np.zeros(n_comp)
            s_all[cand] = index_scores(indexer_query(q_idx[l], idx_fp4), w[l], key_vals[cand])
            idx[l] = topk_set(s_all, topk, candidates=cand)
        else:
            idx[l] = idx[idx_src[l]].copy()
    outs = []
    for l in range(L):
        data, scale, fmt = kv[kv_src[l]]
        wdata, wscale = win[kv_src[l]]
        outs.append(csa_sparse_attention(q[l], data, scale, fmt, idx[l], wdata, wscale,
                                         win_len, tau))
    return idx, pool, outs

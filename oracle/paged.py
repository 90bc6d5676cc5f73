"""Paged (block-table) storage of a cache plane (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages allocate every cache dense ("DeepSeek-V4 KV Cache 深度分析", §二:
``kv_cache`` of shape [max_batch, kv_cache_size, 512]; §四: one indexer key
per compressed entry).  A paged plane stores the same entries in pages of
``page_size`` rows; sequence b's logical block j is page
``block_table[b, j]``.  Paging changes where an entry lives, never what is
computed: every result over a paged plane equals the result over the dense
plane holding the same logical entries.  This module maps between the two.
"""

import numpy as np


def row_of(block_table, page_size: int, b: int, pos):
    """Physical row of logical entry (b, pos)."""
    pos = np.asarray(pos, dtype=np.int64)
    return np.asarray(block_table, dtype=np.int64)[b][pos // page_size] * page_size + pos % page_size


def logical_rows(rows, block_table, page_size: int, b: int, n: int):
    """Entries [0, n) of sequence b, in logical order, from a paged array
    ``rows`` [n_pages * page_size, ...]."""
    return np.asarray(rows)[row_of(block_table, page_size, b, np.arange(n))]


def paged_from_dense(dense, block_table, page_size: int, n_pages: int):
    """Paged array [n_pages * page_size, ...] holding dense [B, cap, ...]
    through ``block_table`` [B, cap / page_size] (unreferenced rows zero)."""
    dense = np.asarray(dense)
    B, cap = dense.shape[:2]
    out = np.zeros((n_pages * page_size,) + dense.shape[2:], dtype=dense.dtype)
    for b in range(B):
        out[row_of(block_table, page_size, b, np.arange(cap))] = dense[b]
    return out

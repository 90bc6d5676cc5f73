"""csa_index_topk (through the C ABI) vs the oracle: exact top-k index sets
(ties to the lower index), scores within the f32 accumulation bound, and
the selection exact on the GPU's own scores."""

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from oracle import fp_formats as ff
from oracle import indexer as oi
from tests.helpers import check_topk, ckv, gpu_plane, np32, score_eps

pytestmark = pytest.mark.gpu


def _case(B, n_list, HI, fmt, seed, dup_frac=0.0):
    keys = []
    for b, n in enumerate(n_list):
        k = wl.rms_rows((n, 128), seed * 100 + b, "cuda")
        if dup_frac and n > 10:
            g = torch.Generator().manual_seed(seed + b)
            nd = int(dup_frac * n)
            dst = torch.randperm(n, generator=g)[:nd]
            srcs = torch.randint(0, n, (nd,), generator=g)
            k[dst.cuda()] = k[srcs.cuda()]
        keys.append(k)
    qi = torch.stack([wl.rms_rows((HI, 128), seed * 1000 + b, "cuda") for b in range(B)])
    w = torch.stack([wl.head_weights((HI,), seed * 7 + b, "cuda") for b in range(B)])
    cap = max(n_list) + 5
    plane = gpu_plane(fmt, 128, keys, cap)
    return keys, qi, w, plane


def _oracle_scores(keys_b, qi_b, w_b, fmt):
    kv = ff.dequantize_entries(*ff.quantize_entries(np32(keys_b), fmt), fmt)
    qv = oi.indexer_query(np32(qi_b), fmt == "fp4")
    w = np32(w_b).astype(np.float64)
    return oi.index_scores(qv, w, kv), score_eps(qv, w, kv)


def _gpu_selection_of(dbg_row, n, k):
    s = dbg_row[:n].astype(np.float64)
    s = np.where(s == 0, 0.0, s)
    return oi.topk_set(s, k)


@pytest.mark.parametrize("fmt,HI,n_list,topk", [
    ("bf16", 4, [1024], 512),                      # the tiny BF16 workload shape
    ("fp4", 64, [3000, 1500, 700], 512),           # ragged, one sequence below... above k
    ("fp4", 64, [300, 9000], 512),                 # n_comp < k: -1 padding
    ("fp4", 64, [0, 5000, 1], 512),                # a sequence with no entries, one with one
    ("fp4", 16, [20000], 1024),                    # several chunks, k = 1024
    ("fp4", 64, [140000, 133000], 512),            # the long-sequence kernel instance
    ("bf16", 8, [5000, 17], 64),
    ("bf16", 16, [2000], 256),                     # CUDA-core scorer sized for 16 heads
    ("bf16", 32, [1500, 900], 128),                # ... for 32 heads
    ("bf16", 64, [800], 512),                      # ... for 64 heads, one chunk
])
def test_index_topk_matches_oracle(fmt, HI, n_list, topk):
    b = ckv()
    B = len(n_list)
    keys, qi, w, plane = _case(B, n_list, HI, fmt, seed=len(n_list) * 31 + HI + topk)
    n_comp = torch.tensor(n_list, dtype=torch.int32, device="cuda")
    n_max = max(n_list)
    dbg = torch.full((B, n_max), float("nan"), device="cuda")
    idx = b.csa_index_topk(plane, n_comp, n_max, qi, w, topk, dbg_scores=dbg)
    torch.cuda.synchronize()
    idx = idx.cpu().numpy()
    dbg = dbg.cpu().numpy()
    for s in range(B):
        sc, eps = _oracle_scores(keys[s], qi[s], w[s], fmt)
        n = n_list[s]
        err = np.abs(dbg[s, :n] - sc)
        assert np.all(err <= eps + 1e-30), "score error %g > bound" % (err / np.maximum(eps, 1e-30)).max()
        assert np.array_equal(idx[s], _gpu_selection_of(dbg[s], n, topk)), "selection on GPU scores"
        assert check_topk(idx[s], sc, eps, topk, where="seq %d" % s) == 0


def test_index_topk_exact_ties_go_to_lower_index():
    """Duplicated key vectors quantise to identical bytes, so their scores tie
    exactly (bitwise on the GPU too); the boundary must go to lower indices."""
    b = ckv()
    n = 6000
    keys, qi, w, plane = _case(1, [n], 64, "fp4", seed=77, dup_frac=0.3)
    # crowd the boundary: copy the entries ranked around 512 many times
    sc, _ = _oracle_scores(keys[0], qi[0], w[0], "fp4")
    order = np.lexsort((np.arange(n), -sc))
    k2 = wl.inject_ties(keys[0], order, seed=3, frac=0.2, donor_lo=500, donor_hi=520)
    plane = gpu_plane("fp4", 128, [k2], n)
    sc, eps = _oracle_scores(k2, qi[0], w[0], "fp4")
    n_comp = torch.tensor([n], dtype=torch.int32, device="cuda")
    dbg = torch.zeros((1, n), device="cuda")
    idx = b.csa_index_topk(plane, n_comp, n, qi, w, 512, dbg_scores=dbg).cpu().numpy()[0]
    d = dbg.cpu().numpy()[0]
    kb = plane.data.cpu().numpy()[0]
    # identical bytes -> identical f32 scores
    _, inv = np.unique(np.concatenate([kb, plane.scale.cpu().numpy()[0]], axis=1), axis=0,
                       return_inverse=True)
    for g in np.unique(inv):
        members = np.nonzero(inv == g)[0]
        assert len(set(d[members].tolist())) == 1
    boundary = sc[oi.topk_set(sc, 512)].min()
    assert (sc == boundary).sum() > 1, "the test must put an exact tie on the boundary"
    assert np.array_equal(idx, oi.topk_set(sc, 512))
    assert np.array_equal(idx, _gpu_selection_of(d, n, 512))


def test_index_long_sequence_exact_ties():
    """The long-sequence kernel instance (more than 131 072 entries) on keys
    whose ranks 481-544 are copied onto 5 % of the other entries: thousands
    of staged candidates, exact ties across the top-512 boundary."""
    b = ckv()
    n = 140000
    keys, qi, w, plane = _case(1, [n], 64, "fp4", seed=81)
    sc, _ = _oracle_scores(keys[0], qi[0], w[0], "fp4")
    order = np.lexsort((np.arange(n), -sc))
    k2 = wl.inject_ties(keys[0], order, seed=4, frac=0.05, donor_lo=480, donor_hi=544)
    plane = gpu_plane("fp4", 128, [k2], n)
    sc, eps = _oracle_scores(k2, qi[0], w[0], "fp4")
    n_comp = torch.tensor([n], dtype=torch.int32, device="cuda")
    dbg = torch.zeros((1, n), device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_INDEX_TOPK, 1, 0, 64, n, 512, 0))
    for _ in range(2):    # the second call checks that the workspace was left clean
        idx = b.csa_index_topk(plane, n_comp, n, qi, w, 512, dbg_scores=dbg, ws=ws).cpu().numpy()[0]
        assert b.read_device_status(ws) == 0
        d = dbg.cpu().numpy()[0]
        assert np.array_equal(idx, _gpu_selection_of(d, n, 512))
        assert check_topk(idx, sc, eps, 512, where="long ties") == 0


@pytest.mark.parametrize("fmt,HI,n_hi,group", [
    ("fp4", 64, 490, 40),     # the merge ranks a short boundary list directly
    ("fp4", 64, 200, 600),    # ... and radix-selects a longer one
    ("bf16", 8, 200, 600),    # the CUDA-core scorer's merge
])
def test_index_boundary_tie_group(fmt, HI, n_hi, group):
    """Three key vectors, each repeated: n_hi copies score highest, `group`
    copies tie exactly on the top-512 boundary, the rest score lowest.  The
    selection is the n_hi plus the group's lowest entries, whatever chunk
    each copy sits in."""
    b = ckv()
    n, k = 3000, 512
    assert n_hi < k < n_hi + group
    base = wl.rms_rows((3, 128), 91, "cuda")
    qi = wl.rms_rows((1, HI, 128), 92, "cuda")
    w = wl.head_weights((1, HI), 93, "cuda")
    sc3, _ = _oracle_scores(base, qi[0], w[0], fmt)
    hi, mid, lo = np.argsort(-sc3)
    assert sc3[hi] > sc3[mid] > sc3[lo]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(94)).numpy()
    which = np.full(n, lo)
    which[perm[:n_hi]] = hi
    which[perm[n_hi:n_hi + group]] = mid
    keys = base[torch.as_tensor(which, device="cuda")]
    plane = gpu_plane(fmt, 128, [keys], n)
    n_comp = torch.tensor([n], dtype=torch.int32, device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_INDEX_TOPK, 1, 0, HI, n, k, 0))
    want = np.sort(np.concatenate([perm[:n_hi], np.sort(perm[n_hi:n_hi + group])[:k - n_hi]]))
    for _ in range(2):    # the second call checks that the workspace was left clean
        idx = b.csa_index_topk(plane, n_comp, n, qi, w, k, ws=ws).cpu().numpy()[0]
        assert b.read_device_status(ws) == 0
        assert np.array_equal(idx, want)


@pytest.mark.parametrize("HI2", [64, 40])
def test_index_pool_and_reindex(HI2):
    """CSA2 Full (pool of 2048 + top-512) then Reindex over that pool: the
    Reindex gathers the pool's key rows into the block-scaled scorer, and a
    head count that is not a multiple of 32 is covered too."""
    b = ckv()
    n = 12000
    keys, qi, w, plane = _case(2, [n, n - 999], 64, "fp4", seed=5)
    n_comp = torch.tensor([n, n - 999], dtype=torch.int32, device="cuda")
    idx, pool = b.csa_index_topk(plane, n_comp, n, qi, w, 512, pool_out=2048)
    qi2 = torch.stack([wl.rms_rows((HI2, 128), 4242 + s, "cuda") for s in range(2)])
    w2 = torch.stack([wl.head_weights((HI2,), 99 + s, "cuda") for s in range(2)])
    dbg = torch.full((2, n), float("nan"), device="cuda")
    idx2 = b.csa_index_topk(plane, n_comp, n, qi2, w2, 512, pool=pool, dbg_scores=dbg)
    torch.cuda.synchronize()
    idx, pool, idx2 = idx.cpu().numpy(), pool.cpu().numpy(), idx2.cpu().numpy()
    dbg = dbg.cpu().numpy()
    for s in range(2):
        sc, eps = _oracle_scores(keys[s], qi[s], w[s], "fp4")
        assert check_topk(pool[s], sc, eps, 2048, where="pool") == 0
        assert check_topk(idx[s], sc, eps, 512, where="full") == 0
        sc2, eps2 = _oracle_scores(keys[s], qi2[s], w2[s], "fp4")
        cand = pool[s][pool[s] >= 0]
        err = np.abs(dbg[s, cand] - sc2[cand])
        assert np.all(err <= eps2[cand] + 1e-30), "reindex score error above the bound"
        assert check_topk(idx2[s], sc2, eps2, 512, candidates=pool[s], where="reindex") == 0
        assert set(idx2[s]) <= set(pool[s])


@pytest.mark.parametrize("n_hi,group", [
    (200, 1200),     # pool boundary among distinct keys, top-512 boundary in a long tie
    (1500, 1200),    # pool boundary in a long tie (top-512 inside the n_hi copies)
])
def test_index_pool_with_crowded_boundary(n_hi, group):
    """CSA2 Full layer (pool of 2048 + top-512) on keys where a boundary falls
    in a run of identical keys longer than the merge's boundary list: n_hi
    copies of the best-scoring key, `group` copies of the second best, the
    rest distinct.  Both outputs must equal the oracle's (ties to the lower
    entries), with the workspace left clean for a second call."""
    b = ckv()
    n, k, P = 12000, 512, 2048
    base = wl.rms_rows((n, 128), 95, "cuda")
    qi = wl.rms_rows((1, 64, 128), 96, "cuda")
    w = wl.head_weights((1, 64), 97, "cuda")
    sc0, _ = _oracle_scores(base, qi[0], w[0], "fp4")
    best, second = np.argsort(-sc0)[:2]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(98)).numpy()
    which = np.arange(n)
    which[perm[:n_hi]] = best
    which[perm[n_hi:n_hi + group]] = second
    keys = base[torch.as_tensor(which, device="cuda")]
    sc, eps = _oracle_scores(keys, qi[0], w[0], "fp4")
    plane = gpu_plane("fp4", 128, [keys], n)
    n_comp = torch.tensor([n], dtype=torch.int32, device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_INDEX_TOPK, 1, 0, 64, n, k, P))
    for _ in range(2):
        idx, pool = b.csa_index_topk(plane, n_comp, n, qi, w, k, pool_out=P, ws=ws)
        assert b.read_device_status(ws) == 0
        idx, pool = idx.cpu().numpy()[0], pool.cpu().numpy()[0]
        assert check_topk(pool, sc, eps, P, where="pool") == 0
        assert check_topk(idx, sc, eps, k, where="top-k") == 0


def test_index_out_of_range_pool_entry_is_flagged():
    b = ckv()
    keys, qi, w, plane = _case(1, [100], 8, "fp4", seed=9)
    n_comp = torch.tensor([100], dtype=torch.int32, device="cuda")
    pool = torch.tensor([[5, 7, 250, -1, 9]], dtype=torch.int32, device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_INDEX_TOPK, 1, 0, 8, 100, 2, 0))
    idx = b.csa_index_topk(plane, n_comp, 100, qi, w, 2, pool=pool, ws=ws)
    assert b.read_device_status(ws) == -6
    sc, _ = _oracle_scores(keys[0], qi[0], w[0], "fp4")
    assert list(idx.cpu().numpy()[0]) == list(oi.topk_set(sc, 2, candidates=[5, 7, 9]))


@pytest.mark.parametrize("fmt,HI,n,topk,pool_out", [
    ("fp4", 64, 20000, 512, 0),       # tensor-core scorer: more equal keys than its merge buffer
    ("fp4", 64, 20000, 512, 2048),    # ... with the CSA2 Full layer's pool
    ("bf16", 8, 20000, 512, 0),       # CUDA-core scorer
    ("fp4", 64, 3000, 512, 0),        # equal keys that still fit the merge buffer
])
def test_index_all_equal_scores_take_the_lowest_entries(fmt, HI, n, topk, pool_out):
    """A zero indexer query makes every score 0: every key ties, the whole
    sequence lands in one histogram bin, and the top-k must be the lowest
    entries (the merge's crowded-boundary path when they outnumber its
    shared-memory buffer)."""
    b = ckv()
    keys = [wl.rms_rows((n, 128), 77, "cuda")]
    plane = gpu_plane(fmt, 128, keys, n)
    qi = torch.zeros((1, HI, 128), dtype=torch.bfloat16, device="cuda")
    w = wl.head_weights((1, HI), 78, "cuda")
    n_comp = torch.tensor([n], dtype=torch.int32, device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_INDEX_TOPK, 1, 0, HI, n, topk, pool_out))
    for _ in range(2):    # the second call checks that the workspace was left clean
        res = b.csa_index_topk(plane, n_comp, n, qi, w, topk, pool_out=pool_out, ws=ws)
        assert b.read_device_status(ws) == 0
        idx = (res[0] if pool_out else res).cpu().numpy()[0]
        assert np.array_equal(idx, np.arange(topk))
        if pool_out:
            assert np.array_equal(res[1].cpu().numpy()[0], np.arange(pool_out))


def test_index_reused_workspace_ignores_earlier_candidates():
    """One workspace, two Reindex calls over 32 pool chunks of 256 entries.
    The first (every pool entry valid, scores 1000x larger) leaves large keys
    in every candidate slot.  In the second, chunk j ends in 1 + j % 3 empty
    (-1) entries: every chunk's list (all its valid keys: each chunk holds
    fewer than top-k) has a length that is not a multiple of 4 and ends on
    the same lane, and 32 lists are more than the merge has warps, so one
    lane stages the last group of several lists.  The earlier call's keys in
    the slots past each list must not count."""
    b = ckv()
    n = 20000
    keys, qi, w, plane = _case(1, [n], 64, "fp4", seed=21)
    n_comp = torch.tensor([n], dtype=torch.int32, device="cuda")
    P = 32 * 256
    ws = b.new_workspace(b.workspace_bytes(b.OP_INDEX_TOPK, 1, 0, 64, n, 512, 0) +
                         b.workspace_bytes(b.OP_INDEX_TOPK, 1, 0, 64, n, 512, P))
    pool1 = torch.arange(P, dtype=torch.int32, device="cuda").view(1, P)
    b.csa_index_topk(plane, n_comp, n, qi, w * 1000.0, 512, pool=pool1, ws=ws)
    pool2 = (torch.arange(P, dtype=torch.int32) * 2 + 1).view(32, 256)
    for j in range(32):
        pool2[j, 256 - (1 + j % 3):] = -1
    pool2 = pool2.reshape(1, P).cuda()
    idx = b.csa_index_topk(plane, n_comp, n, qi, w, 512, pool=pool2, ws=ws)
    assert b.read_device_status(ws) == 0
    sc, eps = _oracle_scores(keys[0], qi[0], w[0], "fp4")
    cand = pool2.cpu().numpy()[0]
    assert check_topk(idx.cpu().numpy()[0], sc, eps, 512, candidates=cand, where="reused workspace") == 0

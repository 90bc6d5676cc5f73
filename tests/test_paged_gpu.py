"""Paged (block-table) cache planes through the C ABI.  Paging changes only
where entries live: every call over a paged plane must give exactly (bit for
bit) what it gives over the dense plane holding the same logical entries,
and the paged append must store the oracle's bytes at the table's rows."""

import math

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from oracle import fp_formats as ff
from oracle import paged as opaged
from tests.helpers import ckv, gpu_plane, np32

pytestmark = pytest.mark.gpu
TAU = 1.0 / math.sqrt(512)


def plane_pair(fmt, dim, rows, cap, page_size, nope_block=448, seed=0):
    """(dense, paged) planes with the same logical entries; the paged one's
    pages are a random permutation with a few spare pages."""
    b = ckv()
    B = len(rows)
    dense = gpu_plane(fmt, dim, rows, cap, nope_block)
    blocks = cap // page_size
    n_pages = B * blocks + 3
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(n_pages, generator=g)[:B * blocks].reshape(B, blocks).to(torch.int32).cuda()
    paged = b.Plane(fmt, dim, B, cap, "cuda", nope_block, block_table=table, page_size=page_size,
                    n_pages=n_pages)
    src, slots = [], []
    for s, r in enumerate(rows):
        if r is None or r.shape[0] == 0:
            continue
        src.append(r)
        slots.append(paged.slot(s, torch.arange(r.shape[0], device="cuda")))
    ws = b.new_workspace(256)
    b.kv_append_quant(paged, torch.cat(src).contiguous(), torch.cat(slots).contiguous(), ws=ws)
    assert b.read_device_status(ws) == 0
    return dense, paged


@pytest.mark.parametrize("fmt,dim", [("fp4", 128), ("fp4h", 128), ("mixed", 512), ("fp4", 512)])
def test_paged_append_stores_the_oracle_bytes(fmt, dim):
    rows = [wl.rms_rows((300, dim), 3000 + s, "cuda") for s in range(2)]
    _, paged = plane_pair(fmt, dim, rows, 512, 256, seed=1)
    table = paged.block_table.cpu().numpy()
    data = paged.data.cpu().numpy()
    scale = None if paged.scale is None else paged.scale.cpu().numpy()
    for s in range(2):
        d, sc = ff.quantize_entries(np32(rows[s]), fmt)
        assert np.array_equal(opaged.logical_rows(data, table, 256, s, 300), d)
        if sc is not None:
            assert np.array_equal(opaged.logical_rows(scale, table, 256, s, 300), sc)


@pytest.mark.parametrize("fmt,HI,n_list,topk,pool_out,page", [
    ("fp4", 64, [9000, 3000], 512, 0, 256),       # tensor-core scorer
    ("fp4", 64, [12000, 5000], 512, 2048, 128),   # with the CSA2 Full pool
    ("fp4h", 32, [7000], 256, 0, 512),
    ("bf16", 8, [5000, 1200], 512, 0, 128),       # CUDA-core scorer
])
def test_paged_index_topk_equals_dense(fmt, HI, n_list, topk, pool_out, page):
    b = ckv()
    B = len(n_list)
    cap = (max(n_list) + page - 1) // page * page
    keys = [wl.rms_rows((n, 128), 3100 + s, "cuda") for s, n in enumerate(n_list)]
    dense, paged = plane_pair(fmt, 128, keys, cap, page, seed=2)
    qi = wl.rms_rows((B, HI, 128), 3200, "cuda")
    w = wl.head_weights((B, HI), 3201, "cuda")
    n_comp = torch.tensor(n_list, dtype=torch.int32, device="cuda")
    d = b.csa_index_topk(dense, n_comp, max(n_list), qi, w, topk, pool_out=pool_out)
    p = b.csa_index_topk(paged, n_comp, max(n_list), qi, w, topk, pool_out=pool_out)
    torch.cuda.synchronize()
    if pool_out:
        assert torch.equal(d[0], p[0]) and torch.equal(d[1], p[1])
        # Reindex over the pool of a paged plane (CUDA-core scorer, per-key pages)
        qi2 = wl.rms_rows((B, HI, 128), 3202, "cuda")
        assert torch.equal(b.csa_index_topk(dense, n_comp, max(n_list), qi2, w, topk, pool=d[1]),
                           b.csa_index_topk(paged, n_comp, max(n_list), qi2, w, topk, pool=p[1]))
    else:
        assert torch.equal(d, p)


@pytest.mark.parametrize("fmt,H,page", [("mixed", 128, 128), ("fp4", 64, 256), ("bf16", 128, 128)])
def test_paged_csa_attention_equals_dense(fmt, H, page):
    b = ckv()
    B, n, W, topk = 2, 3000, 128, 512
    cap = (n + page - 1) // page * page
    kv = [wl.rms_rows((n, 512), 3300 + s, "cuda") for s in range(B)]
    win = [wl.rms_rows((W, 512), 3400 + s, "cuda") for s in range(B)]
    dense, paged = plane_pair(fmt, 512, kv, cap, page, seed=3)
    wp = gpu_plane(fmt, 512, win, W)
    q = wl.rms_rows((B, H, 512), 3500, "cuda")
    g = torch.Generator().manual_seed(5)
    idx = torch.stack([torch.sort(torch.randperm(n, generator=g)[:topk])[0] for _ in range(B)]).to(torch.int32).cuda()
    idx[0, 7] = -1
    wlen = torch.tensor([W, 33], dtype=torch.int32, device="cuda")
    l1, l2 = torch.empty((B, H), device="cuda"), torch.empty((B, H), device="cuda")
    o1 = b.csa_sparse_attn(dense, wp, wlen, idx, q, TAU, lse=l1)
    o2 = b.csa_sparse_attn(paged, wp, wlen, idx, q, TAU, lse=l2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("fmt,n", [("bf16", 8320), ("mixed", 1000)])
def test_paged_hca_attention_equals_dense(fmt, n):
    b = ckv()
    B, H, W, page = 2, 128, 128, 128
    cap = (n + page - 1) // page * page
    kv = [wl.rms_rows((n, 512), 3600 + s, "cuda") for s in range(B)]
    win = [wl.rms_rows((W, 512), 3700 + s, "cuda") for s in range(B)]
    dense, paged = plane_pair(fmt, 512, kv, cap, page, seed=4)
    wp = gpu_plane(fmt, 512, win, W)
    q = wl.rms_rows((B, H, 512), 3800, "cuda")
    n_comp = torch.tensor([n, n - 77], dtype=torch.int32, device="cuda")
    wlen = torch.full((B,), W, dtype=torch.int32, device="cuda")
    l1, l2 = torch.empty((B, H), device="cuda"), torch.empty((B, H), device="cuda")
    o1 = b.hca_attn(dense, n_comp, n, wp, wlen, q, TAU, lse=l1)
    o2 = b.hca_attn(paged, n_comp, n, wp, wlen, q, TAU, lse=l2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_paged_csa2_group_equals_dense():
    b = ckv()
    B, n, H, HI, topk, W, L, P, page = 2, 2300, 64, 64, 64, 128, 3, 256, 256
    cap = (n + 16 + page - 1) // page * page
    keys = [wl.rms_rows((n, 128), 3900 + s, "cuda") for s in range(B)]
    kvs = [[wl.rms_rows((n, 512), 4000 + 10 * l + s, "cuda") for s in range(B)] for l in range(L)]
    wins = [[wl.rms_rows((W, 512), 4100 + 10 * l + s, "cuda") for s in range(B)] for l in range(L)]
    kd, kp = plane_pair("fp4", 128, keys, cap, page, seed=6)
    pairs = [plane_pair("fp4", 512, kvs[l], cap, page, seed=7 + l) for l in range(L)]
    wp = [gpu_plane("fp4", 512, wins[l], W) for l in range(L)]
    q = [wl.rms_rows((B, H, 512), 4200 + l, "cuda") for l in range(L)]
    qi = [wl.rms_rows((B, HI, 128), 4300, "cuda"), wl.rms_rows((B, HI, 128), 4301, "cuda"), None]
    w = [wl.head_weights((B, HI), 4302, "cuda"), wl.head_weights((B, HI), 4303, "cuda"), None]
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    wlen = torch.full((B,), W, dtype=torch.int32, device="cuda")
    roles = [b.CSA2_FULL, b.CSA2_REINDEX, b.CSA2_REUSE]
    app = wl.rms_rows((16, 512), 4400, "cuda")
    outs = []
    for which in (0, 1):
        out = [torch.empty_like(q[0]) for _ in range(L)]
        kvl = [pairs[l][which] for l in range(L)]
        g = b.make_group(roles, [0, 0, 2], [0, 0, 0], kvl, wp, (kd, kp)[which], q, qi, w, out, pool_len=P)
        slot = torch.cat([kvl[0].slot(s, torch.arange(n, n + 8, device="cuda")) for s in range(B)]).to(torch.int64)
        ws = b.csa2_group_decode(g, n_comp, n, wlen, B, H, HI, topk, TAU, append_dst=kvl[0],
                                 append_src=app, append_slot=slot)
        assert b.read_device_status(ws) == 0
        outs.append(out)
    for l in range(L):
        assert torch.equal(outs[0][l], outs[1][l])

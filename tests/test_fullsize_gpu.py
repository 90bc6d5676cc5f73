"""Parity at the full workload sizes, in the launch configuration bench.py
times (same batch, entry counts, heads, formats), on sampled sequences the
oracle computes one by one."""

import math

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wlmod
from oracle import attention as oa
from oracle import csa2 as oc
from oracle import fp_formats as ff
from oracle import indexer as oi
from tests.helpers import check_attention, check_topk, ckv, np32, score_eps

pytestmark = pytest.mark.gpu


def _fill(b, plane, rows, seq, cap):
    b.kv_append_quant(plane, rows, torch.arange(rows.shape[0], dtype=torch.int64, device="cuda") + seq * cap)


@pytest.mark.parametrize("name,sample", [("csa_tiny_4k", [0]), ("csa_128k", [0, 5]), ("csa_1m", [2]),
                                         ("csa_128k_pro", [3])])
def test_csa_full_size(name, sample):
    b = ckv()
    wl = wlmod.WORKLOADS[name]
    B, n, cap = wl.B, wl.n_comp, wl.n_comp + 8
    kv = b.Plane(wl.main_fmt, 512, B, cap, nope_block=wl.nope_block)
    win = b.Plane(wl.main_fmt, 512, B, wl.W, nope_block=wl.nope_block)
    keys = b.Plane(wl.idx_fmt, 128, B, cap)
    q, qi, w = wlmod.step_queries(wl, 0, "cuda")
    rows = {}
    for s in range(B):
        kvr, kr, wr = wlmod.sequence_rows(wl, s, n, "cuda")
        if wl.ties and s in sample:
            # ties crowded at the boundary, ranked by the oracle's scores
            kvals = ff.dequantize_entries(*ff.quantize_entries(np32(kr), wl.idx_fmt), wl.idx_fmt)
            sc = oi.index_scores(oi.indexer_query(np32(qi[s]), True), np32(w[s]).astype(np.float64), kvals)
            kr = wlmod.inject_ties(kr, np.lexsort((np.arange(n), -sc)), seed=wl.seed + s)
        _fill(b, kv, kvr, s, cap)
        _fill(b, keys, kr, s, cap)
        _fill(b, win, wr, s, wl.W)
        if s in sample:
            rows[s] = (kvr.cpu(), kr.cpu(), wr.cpu())
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    win_len = torch.full((B,), wl.W, dtype=torch.int32, device="cuda")
    ws = b.new_workspace(max(b.workspace_bytes(b.OP_INDEX_TOPK, B, wl.H, wl.HI, n, wl.topk, 0),
                             b.workspace_bytes(b.OP_SPARSE_ATTN, B)))
    idx = b.csa_index_topk(keys, n_comp, n, qi, w, wl.topk, ws=ws)
    lse = torch.empty((B, wl.H), device="cuda")
    out = b.csa_sparse_attn(kv, win, win_len, idx, q, wl.tau, lse=lse, ws=ws)
    assert b.read_device_status(ws) == 0
    ties_seen = 0
    for s in sample:
        kvr, kr, wr = rows[s]
        kvals = ff.dequantize_entries(*ff.quantize_entries(np32(kr), wl.idx_fmt), wl.idx_fmt)
        qv = oi.indexer_query(np32(qi[s]), wl.idx_fmt == "fp4")
        ww = np32(w[s]).astype(np.float64)
        sc = oi.index_scores(qv, ww, kvals)
        eps = score_eps(qv, ww, kvals)
        got = idx[s].cpu().numpy()
        assert check_topk(got, sc, eps, wl.topk, where="%s seq %d" % (name, s)) == 0
        want = oi.topk_set(sc, wl.topk)
        ties_seen += int((sc == sc[want].min()).sum() > 1)
        sel = want[want >= 0]
        kd, ks = ff.quantize_entries(np32(kvr)[sel], wl.main_fmt, wl.nope_block)
        wd, wsc = ff.quantize_entries(np32(wr), wl.main_fmt, wl.nope_block)
        o_ref, l_ref = oa.csa_sparse_attention(np32(q[s]), kd, ks, wl.main_fmt, np.arange(len(sel)),
                                               wd, wsc, wl.W, wl.tau, nope_block=wl.nope_block)
        check_attention(out[s], lse[s], o_ref, l_ref, wl.H, where="%s seq %d" % (name, s))
    if wl.ties:
        assert ties_seen == len(sample), "tie injection must put exact ties on the boundary"


def test_hca_full_size():
    b = ckv()
    wl = wlmod.WORKLOADS["hca_1m"]
    B, n, cap = wl.B, wl.n_comp, wl.n_comp + 8
    kv = b.Plane("bf16", 512, B, cap)
    win = b.Plane("bf16", 512, B, wl.W)
    q, _, _ = wlmod.step_queries(wl, 0, "cuda")
    rows = {}
    sample = [0, 11, 15]
    for s in range(B):
        kvr, _, wr = wlmod.sequence_rows(wl, s, n, "cuda")
        _fill(b, kv, kvr, s, cap)
        _fill(b, win, wr, s, wl.W)
        if s in sample:
            rows[s] = (kvr.cpu(), wr.cpu())
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    win_len = torch.full((B,), wl.W, dtype=torch.int32, device="cuda")
    lse = torch.empty((B, wl.H), device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_HCA_ATTN, B))
    out = b.hca_attn(kv, n_comp, n, win, win_len, q, wl.tau, lse=lse, ws=ws)
    assert b.read_device_status(ws) == 0
    for s in sample:
        kvr, wr = rows[s]
        o_ref, l_ref = oa.hca_attention(np32(q[s]), ff.bf16_bytes(np32(kvr)), None, "bf16", n,
                                        ff.bf16_bytes(np32(wr)), None, wl.W, wl.tau)
        check_attention(out[s], lse[s], o_ref, l_ref, wl.H, where="hca_1m seq %d" % s)


def test_csa2_full_size():
    b = ckv()
    wl = wlmod.WORKLOADS["csa2_group"]
    B, n, L, cap = wl.B, wl.n_comp, wl.n_layers, wl.n_comp + 16
    s0 = 3
    keys = b.Plane("fp4", 128, B, cap)
    kvs = [b.Plane("fp4", 512, B, cap) for _ in range(L)]
    wins = [b.Plane("fp4", 512, B, wl.W) for _ in range(L)]
    keep = {}
    for l in range(L):
        for s in range(B):
            kvr, kr, wr = wlmod.sequence_rows(wl, s, n, "cuda", layer=l)
            _fill(b, kvs[l], kvr, s, cap)
            _fill(b, wins[l], wr, s, wl.W)
            if l == 0:
                _fill(b, keys, kr, s, cap)
            if s == s0:
                keep[l] = (kvr.cpu(), kr.cpu() if l == 0 else None, wr.cpu())
    qs, qis, wss = [], [], []
    for l in range(L):
        ql, qil, wl_ = wlmod.step_queries(wl, 0, "cuda", layer=l)
        qs.append(ql)
        qis.append(qil if l < 2 else None)
        wss.append(wl_ if l < 2 else None)
    outs = [torch.empty_like(qs[0]) for _ in range(L)]
    lses = [torch.empty((B, wl.H), device="cuda") for _ in range(L)]
    idx_out = [torch.empty((B, wl.topk), dtype=torch.int32, device="cuda") for _ in range(L)]
    roles = [oc.FULL, oc.REINDEX] + [oc.REUSE] * (L - 2)
    kv_src, idx_src = [0, 0] + list(range(2, L)), [0] * L
    g = b.make_group(roles, kv_src, idx_src, kvs, wins, keys, qs, qis, wss, outs, lse=lses,
                     idx_out=idx_out, pool_len=wl.pool_len)
    app = wlmod.append_rows(wl, wl.n_append, 512, 0, "cuda")
    per = wl.n_append // B
    slot = (torch.arange(B)[:, None] * cap + n + torch.arange(per)[None]).flatten().to(torch.int64).cuda()
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    win_len = torch.full((B,), wl.W, dtype=torch.int32, device="cuda")
    ws = b.csa2_group_decode(g, n_comp, n, win_len, B, wl.H, wl.HI, wl.topk, wl.tau, append_dst=kvs[0],
                             append_src=app, append_slot=slot)
    assert b.read_device_status(ws) == 0
    kd, ks = ff.fp4_quantize(np32(keep[0][1]))
    kvals = ff.fp4_dequantize(kd, ks)
    qi_np = [np32(qis[l][s0]) if qis[l] is not None else None for l in range(L)]
    w_np = [np32(wss[l][s0]).astype(np.float64) if wss[l] is not None else None for l in range(L)]
    # index sets
    gi = [idx_out[l][s0].cpu().numpy() for l in range(L)]
    qv0 = oi.indexer_query(qi_np[0], True)
    sc0 = oi.index_scores(qv0, w_np[0], kvals)
    assert check_topk(gi[0], sc0, score_eps(qv0, w_np[0], kvals), wl.topk, where="full") == 0
    pool = oi.topk_set(sc0, wl.pool_len)
    qv1 = oi.indexer_query(qi_np[1], True)
    sc1 = oi.index_scores(qv1, w_np[1], kvals)
    assert check_topk(gi[1], sc1, score_eps(qv1, w_np[1], kvals), wl.topk, candidates=pool,
                      where="reindex") == 0
    # attention of every layer on the gathered rows only
    for l in range(L):
        src = kv_src[l]
        idx_l = gi[l] if l < 2 else gi[0]
        kvr, _, wr = keep[src]
        kd, ks = ff.fp4_quantize(np32(kvr)[idx_l])
        wd, wsc = ff.fp4_quantize(np32(wr))
        o_ref, l_ref = oa.csa_sparse_attention(np32(qs[l][s0]), kd, ks, "fp4", np.arange(len(idx_l)),
                                               wd, wsc, wl.W, wl.tau)
        check_attention(outs[l][s0], lses[l][s0], o_ref, l_ref, wl.H, where="csa2 layer %d" % l)

"""csa_sparse_attn / hca_attn (through the C ABI) vs the float64 oracle:
max |err| <= 2e-2 and per-head relative error <= 1e-2 on the bf16 output,
lse within 1e-2."""

import math

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from oracle import attention as oa
from tests.helpers import check_attention, ckv, gpu_plane, np32, oracle_plane

pytestmark = pytest.mark.gpu
TAU = 1.0 / math.sqrt(512)


def _seq_rows(B, n_list, W, seed, spikes=False):
    kv = [wl.rms_rows((n, 512), seed * 10 + b, "cuda", spikes=spikes) for b, n in enumerate(n_list)]
    win = [wl.rms_rows((W, 512), seed * 10 + 5000 + b, "cuda", spikes=spikes) for b in range(B)]
    return kv, win


@pytest.mark.parametrize("fmt,blk,H,n_list,win_lens", [
    ("bf16", 448, 128, [300, 77], [128, 5]),
    ("bf16", 448, 16, [1000], [128]),
    ("mixed", 448, 128, [513, 64], [128, 0]),
    ("mixed", 64, 64, [200], [17]),
    ("fp4", 448, 64, [640, 1], [128, 128]),
    ("bf16", 448, 128, [0, 3], [0, 0]),          # nothing to attend / three rows
    ("bf16", 448, 128, [8192 + 9], [128]),       # many tiles per pair
    # twelve sequences of 32+ tiles: pair clusters fit more CTA pairs than one
    # cluster per sequence, and the last CTA of each half merges
    ("bf16", 448, 16, [2048] * 11 + [2047], [128] * 11 + [3]),
])
def test_hca_matches_oracle(fmt, blk, H, n_list, win_lens):
    b = ckv()
    B, W = len(n_list), 128
    kv, win = _seq_rows(B, n_list, W, seed=sum(n_list) + H)
    cap = max(max(n_list), 1)
    kvp = gpu_plane(fmt, 512, kv, cap, blk)
    wp = gpu_plane(fmt, 512, win, W, blk)
    q = torch.stack([wl.rms_rows((H, 512), 777 + s, "cuda") for s in range(B)])
    n_comp = torch.tensor(n_list, dtype=torch.int32, device="cuda")
    wl_t = torch.tensor(win_lens, dtype=torch.int32, device="cuda")
    lse = torch.empty((B, H), device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_HCA_ATTN, B))
    out = b.hca_attn(kvp, n_comp, max(n_list), wp, wl_t, q, TAU, lse=lse, ws=ws)
    assert b.read_device_status(ws) == 0
    okv, owin = oracle_plane(fmt, kv, blk), oracle_plane(fmt, win, blk)
    for s in range(B):
        o_ref, l_ref = oa.hca_attention(np32(q[s]), okv[s][0], okv[s][1], fmt, n_list[s],
                                        owin[s][0], owin[s][1], win_lens[s], TAU, blk)
        check_attention(out[s], lse[s], o_ref, l_ref, H, where="hca seq %d" % s)


@pytest.mark.parametrize("fmt,blk,H,topk", [
    ("mixed", 448, 128, 512),
    ("mixed", 64, 128, 512),
    ("fp4", 448, 64, 512),
    ("bf16", 448, 16, 512),
    ("mixed", 448, 128, 1024),
    ("fp4", 448, 128, 100),
])
def test_csa_matches_oracle(fmt, blk, H, topk):
    b = ckv()
    B, W, n = 3, 128, 3000
    kv, win = _seq_rows(B, [n] * B, W, seed=topk + H, spikes=fmt == "fp4")
    kvp = gpu_plane(fmt, 512, kv, n, blk)
    wp = gpu_plane(fmt, 512, win, W, blk)
    q = torch.stack([wl.rms_rows((H, 512), 99 + s, "cuda") for s in range(B)])
    g = torch.Generator().manual_seed(topk)
    idx = torch.stack([torch.randperm(n, generator=g)[:topk] for _ in range(B)]).to(torch.int32)
    idx[1, ::7] = -1                    # padding in the middle
    idx[2, 5] = idx[2, 6]               # a duplicate row counts twice
    win_lens = [128, 60, 0]
    wl_t = torch.tensor(win_lens, dtype=torch.int32, device="cuda")
    lse = torch.empty((B, H), device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_SPARSE_ATTN, B))
    out = b.csa_sparse_attn(kvp, wp, wl_t, idx.cuda(), q, TAU, lse=lse, ws=ws)
    assert b.read_device_status(ws) == 0
    okv, owin = oracle_plane(fmt, kv, blk), oracle_plane(fmt, win, blk)
    for s in range(B):
        o_ref, l_ref = oa.csa_sparse_attention(np32(q[s]), okv[s][0], okv[s][1], fmt, idx[s].numpy(),
                                               owin[s][0], owin[s][1], win_lens[s], TAU, blk)
        check_attention(out[s], lse[s], o_ref, l_ref, H, where="csa seq %d" % s)


@pytest.mark.parametrize("fmt", ["mixed", "fp4"])
def test_csa_with_nothing_to_attend(fmt):
    """Every selected index -1: sequence 0 attends its window only, sequence
    1 (window length 0) attends nothing: zero output and lse -inf."""
    b = ckv()
    B, W, n, H, topk = 2, 128, 600, 64, 512
    kv, win = _seq_rows(B, [n] * B, W, seed=41)
    kvp, wp = gpu_plane(fmt, 512, kv, n), gpu_plane(fmt, 512, win, W)
    q = torch.stack([wl.rms_rows((H, 512), 43 + s, "cuda") for s in range(B)])
    idx = torch.full((B, topk), -1, dtype=torch.int32)
    win_lens = [W, 0]
    lse = torch.empty((B, H), device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_SPARSE_ATTN, B))
    out = b.csa_sparse_attn(kvp, wp, torch.tensor(win_lens, dtype=torch.int32, device="cuda"),
                            idx.cuda(), q, TAU, lse=lse, ws=ws)
    assert b.read_device_status(ws) == 0
    okv, owin = oracle_plane(fmt, kv), oracle_plane(fmt, win)
    o_ref, l_ref = oa.csa_sparse_attention(np32(q[0]), okv[0][0], okv[0][1], fmt, idx[0].numpy(),
                                           owin[0][0], owin[0][1], W, TAU)
    check_attention(out[0], lse[0], o_ref, l_ref, H, where="window only")
    assert out[1].float().abs().max().item() == 0.0
    assert bool(torch.isneginf(lse[1]).all())


def test_csa_with_every_entry_equals_hca_on_gpu():
    b = ckv()
    n, W, H = 700, 128, 128
    kv, win = _seq_rows(1, [n], W, seed=3)
    kvp, wp = gpu_plane("mixed", 512, kv, n), gpu_plane("mixed", 512, win, W)
    q = wl.rms_rows((1, H, 512), 5, "cuda")
    wl_t = torch.tensor([W], dtype=torch.int32, device="cuda")
    o_h = b.hca_attn(kvp, torch.tensor([n], dtype=torch.int32, device="cuda"), n, wp, wl_t, q, TAU)
    idx = torch.arange(n, dtype=torch.int32, device="cuda")[None]
    o_c = b.csa_sparse_attn(kvp, wp, wl_t, idx, q, TAU)
    torch.cuda.synchronize()
    assert (o_h.float() - o_c.float()).abs().max().item() <= 2e-2


def test_csa_out_of_range_index_is_flagged():
    b = ckv()
    n, W, H = 100, 128, 16
    kv, win = _seq_rows(1, [n], W, seed=8)
    kvp, wp = gpu_plane("bf16", 512, kv, n), gpu_plane("bf16", 512, win, W)
    q = wl.rms_rows((1, H, 512), 6, "cuda")
    idx = torch.tensor([[3, 500, 7]], dtype=torch.int32, device="cuda")
    wl_t = torch.tensor([4], dtype=torch.int32, device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_SPARSE_ATTN, 1))
    out = b.csa_sparse_attn(kvp, wp, wl_t, idx, q, TAU, ws=ws)
    assert b.read_device_status(ws) == -6
    okv, owin = oracle_plane("bf16", kv), oracle_plane("bf16", win)
    o_ref, l_ref = oa.csa_sparse_attention(np32(q[0]), okv[0][0], None, "bf16", np.array([3, -1, 7]),
                                           owin[0][0], None, 4, TAU)
    check_attention(out[0], None, o_ref, l_ref, H)


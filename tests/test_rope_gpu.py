"""RoPE at the attention's ends ("DeepSeek-V4 KV Cache 深度分析", §五: the query
turned by +i, the core attention output by -i) through the C ABI against the
float64 oracle (oracle.rope), for CSA and HCA in every cache format, small and
1M-scale positions, and the CSA2 group; tolerance as every attention test."""

import math

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from oracle import attention as oa
from oracle import csa2 as oc
from oracle import fp_formats as ff
from oracle import rope as orope
from tests.helpers import check_attention, ckv, gpu_plane, np32, oracle_plane

pytestmark = pytest.mark.gpu
TAU = 1.0 / math.sqrt(512)


def _rope(b, pos, freq, rq, ro):
    p = torch.tensor(pos, dtype=torch.int32, device="cuda")
    f = torch.tensor(freq, dtype=torch.float32, device="cuda")
    return b.Rope(p, f, rq, ro)


@pytest.mark.parametrize("fmt,rq,ro,pos", [
    ("mixed", 1, 1, [131071, 7]),
    ("mixed", 1, 0, [1048575, 0]),
    ("bf16", 0, 1, [5, 999983]),
    ("fp4", 1, 1, [262143, 100000]),
])
def test_csa_rope_matches_oracle(fmt, rq, ro, pos):
    b = ckv()
    B, n, H, W, topk = 2, 1500, 128, 128, 512
    kv = [wl.rms_rows((n, 512), 1300 + s, "cuda") for s in range(B)]
    win = [wl.rms_rows((W, 512), 1400 + s, "cuda") for s in range(B)]
    kvp, wp = gpu_plane(fmt, 512, kv, n), gpu_plane(fmt, 512, win, W)
    q = wl.rms_rows((B, H, 512), 1500, "cuda")
    g = torch.Generator().manual_seed(3)
    idx = torch.stack([torch.sort(torch.randperm(n, generator=g)[:topk])[0] for _ in range(B)]).to(torch.int32).cuda()
    wlen = torch.tensor([W, 50], dtype=torch.int32, device="cuda")
    freq = orope.standard_inv_freq()
    rp = _rope(b, pos, freq, rq, ro)
    lse = torch.empty((B, H), device="cuda")
    out = b.csa_sparse_attn(kvp, wp, wlen, idx, q, TAU, lse=lse, rope=rp)
    okv, owin = oracle_plane(fmt, kv), oracle_plane(fmt, win)
    for s in range(B):
        att = lambda qq: oa.csa_sparse_attention(qq, okv[s][0], okv[s][1], fmt, idx[s].cpu().numpy(),
                                                 owin[s][0], owin[s][1], int(wlen[s]), TAU)
        o_ref, l_ref = orope.attention_with_rope(att, np32(q[s]), pos[s], freq, bool(rq), bool(ro))
        check_attention(out[s], lse[s], o_ref, l_ref, H, where="csa rope seq %d" % s)


@pytest.mark.parametrize("rq,ro", [(1, 1), (0, 1)])
def test_hca_rope_matches_oracle(rq, ro):
    b = ckv()
    B, n, H, W = 2, 3000, 128, 128
    kv = [wl.rms_rows((n, 512), 1600 + s, "cuda") for s in range(B)]
    win = [wl.rms_rows((W, 512), 1700 + s, "cuda") for s in range(B)]
    kvp, wp = gpu_plane("bf16", 512, kv, n), gpu_plane("bf16", 512, win, W)
    q = wl.rms_rows((B, H, 512), 1800, "cuda")
    pos = [1048576 + 3, 4096]
    freq = orope.standard_inv_freq(base=50000.0)
    rp = _rope(b, pos, freq, rq, ro)
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    wlen = torch.full((B,), W, dtype=torch.int32, device="cuda")
    lse = torch.empty((B, H), device="cuda")
    out = b.hca_attn(kvp, n_comp, n, wp, wlen, q, TAU, lse=lse, rope=rp)
    okv, owin = oracle_plane("bf16", kv), oracle_plane("bf16", win)
    for s in range(B):
        att = lambda qq: oa.hca_attention(qq, okv[s][0], okv[s][1], "bf16", n, owin[s][0], owin[s][1], W, TAU)
        o_ref, l_ref = orope.attention_with_rope(att, np32(q[s]), pos[s], freq, bool(rq), bool(ro))
        check_attention(out[s], lse[s], o_ref, l_ref, H, where="hca rope seq %d" % s)


def test_rope_at_position_zero_is_plain_attention():
    b = ckv()
    B, n, H, W = 1, 700, 64, 128
    kv = [wl.rms_rows((n, 512), 1900, "cuda")]
    win = [wl.rms_rows((W, 512), 1901, "cuda")]
    kvp, wp = gpu_plane("mixed", 512, kv, n), gpu_plane("mixed", 512, win, W)
    q = wl.rms_rows((B, H, 512), 1902, "cuda")
    idx = torch.arange(512, dtype=torch.int32, device="cuda")[None]
    wlen = torch.full((B,), W, dtype=torch.int32, device="cuda")
    plain = b.csa_sparse_attn(kvp, wp, wlen, idx, q, TAU)
    rot = b.csa_sparse_attn(kvp, wp, wlen, idx, q, TAU, rope=_rope(b, [0], orope.standard_inv_freq(), 1, 1))
    assert torch.equal(plain, rot)


def test_csa2_group_with_rope():
    b = ckv()
    B, n, H, HI, topk, W, L, P = 2, 2000, 64, 64, 64, 128, 3, 128
    keys = [wl.rms_rows((n, 128), 2000 + s, "cuda") for s in range(B)]
    kvs = [[wl.rms_rows((n, 512), 2100 + 10 * l + s, "cuda") for s in range(B)] for l in range(L)]
    wins = [[wl.rms_rows((W, 512), 2200 + 10 * l + s, "cuda") for s in range(B)] for l in range(L)]
    kplane = gpu_plane("fp4", 128, keys, n)
    kvp = [gpu_plane("fp4", 512, kvs[l], n) for l in range(L)]
    wp = [gpu_plane("fp4", 512, wins[l], W) for l in range(L)]
    q = [wl.rms_rows((B, H, 512), 2300 + l, "cuda") for l in range(L)]
    qi = [wl.rms_rows((B, HI, 128), 2400, "cuda"), wl.rms_rows((B, HI, 128), 2401, "cuda"), None]
    w = [wl.head_weights((B, HI), 2402, "cuda"), wl.head_weights((B, HI), 2403, "cuda"), None]
    out = [torch.empty_like(q[0]) for _ in range(L)]
    lse = [torch.empty((B, H), device="cuda") for _ in range(L)]
    idx_out = [torch.empty((B, topk), dtype=torch.int32, device="cuda") for _ in range(L)]
    pos = [262144 + 17, 91]
    freq = orope.standard_inv_freq()
    roles = [oc.FULL, oc.REINDEX, oc.REUSE]
    g = b.make_group(roles, [0, 0, 2], [0, 0, 0], kvp, wp, kplane, q, qi, w, out, lse=lse, idx_out=idx_out,
                     pool_len=P, rope=_rope(b, pos, freq, 1, 1))
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    wlen = torch.full((B,), W, dtype=torch.int32, device="cuda")
    ws = b.csa2_group_decode(g, n_comp, n, wlen, B, H, HI, topk, TAU)
    assert b.read_device_status(ws) == 0
    for s in range(B):
        okv = [ff.fp4_quantize(np32(kvs[l][s])) for l in range(L)]
        owin = [ff.fp4_quantize(np32(wins[l][s])) for l in range(L)]
        for l in range(L):
            src = [0, 0, 2][l]
            sel = idx_out[l][s].cpu().numpy()
            att = lambda qq: oa.csa_sparse_attention(qq, okv[src][0], okv[src][1], "fp4", sel, owin[src][0],
                                                     owin[src][1], W, TAU)
            o_ref, l_ref = orope.attention_with_rope(att, np32(q[l][s]), pos[s], freq, True, True)
            check_attention(out[l][s], lse[l][s], o_ref, l_ref, H, where="csa2 rope layer %d seq %d" % (l, s))

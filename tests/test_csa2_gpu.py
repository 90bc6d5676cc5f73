"""csa2_group_decode (through the C ABI) vs the oracle's CSA2 wiring."""

import math

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from oracle import csa2 as oc
from oracle import fp_formats as ff
from oracle import indexer as oi
from tests.helpers import check_attention, check_topk, ckv, gpu_plane, np32, oracle_plane, score_eps

pytestmark = pytest.mark.gpu
TAU = 1.0 / math.sqrt(512)


# Every wiring here has a Reindex layer, so the Reindex pass runs beside a
# first attention launch, on the library's side stream, of the layers whose
# indices come from the Full pass: the bench wiring (Reuse of layer 0) as
# launches of four and L - 4 layers, the pages wiring (Reuse of the previous
# layer) as layer 0 alone and then the rest in launches of at most four.
@pytest.mark.parametrize("pool_len,wiring,L", [(256, "bench", 6), (64, "pages", 6),
                                                (64, "degenerate", 6), (64, "pages", 8),
                                                (64, "pages", 5), (64, "pages", 3),
                                                (256, "no_reindex", 5)])
def test_csa2_group_matches_oracle(pool_len, wiring, L):
    b = ckv()
    B, n, H, HI, topk, W = 2, 2500, 64, 64, 64, 128
    if wiring == "degenerate":
        pool_len = topk
    cap = n + 16
    keys = [wl.rms_rows((n, 128), 50 + s, "cuda") for s in range(B)]
    kvs = [[wl.rms_rows((n, 512), 100 * l + s, "cuda", spikes=True) for s in range(B)] for l in range(L)]
    wins = [[wl.rms_rows((W, 512), 1000 + 100 * l + s, "cuda") for s in range(B)] for l in range(L)]
    kplane = gpu_plane("fp4", 128, keys, cap)
    kvp = [gpu_plane("fp4", 512, kvs[l], cap) for l in range(L)]
    wp = [gpu_plane("fp4", 512, wins[l], W) for l in range(L)]
    q = [wl.rms_rows((B, H, 512), 7000 + l, "cuda") for l in range(L)]
    qi = [wl.rms_rows((B, HI, 128), 8000 + l, "cuda") if l < 2 else None for l in range(L)]
    w = [wl.head_weights((B, HI), 9000 + l, "cuda") if l < 2 else None for l in range(L)]
    out = [torch.empty_like(q[0]) for _ in range(L)]
    lse = [torch.empty((B, H), device="cuda") for _ in range(L)]
    idx_out = [torch.empty((B, topk), dtype=torch.int32, device="cuda") for _ in range(L)]
    roles = [oc.FULL, oc.REINDEX] + [oc.REUSE] * (L - 2)
    if wiring == "no_reindex":   # every layer in layer order on the caller's stream
        roles = [oc.FULL] + [oc.REUSE] * (L - 1)
        kv_src, idx_src = list(range(L)), [0] * L
    elif wiring == "bench":
        kv_src, idx_src = [0, 0] + list(range(2, L)), [0] * L
    else:   # the pages' reading: previous layer's indices, one shared KV
        kv_src, idx_src = [0] * L, [0, 0] + list(range(1, L - 1))
    g = b.make_group(roles, kv_src, idx_src, kvp, wp, kplane, q, qi, w, out, lse=lse, idx_out=idx_out,
                     pool_len=pool_len)
    # 16 appended rows (8 per sequence) into layer 0's main KV at [n, n + 8)
    app = wl.rms_rows((16, 512), 31337, "cuda")
    slot = (torch.arange(B)[:, None] * cap + n + torch.arange(8)[None]).flatten().to(torch.int64).cuda()
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    win_len = torch.tensor([W, 77], dtype=torch.int32, device="cuda")
    ws = b.csa2_group_decode(g, n_comp, n, win_len, B, H, HI, topk, TAU, append_dst=kvp[0],
                             append_src=app, append_slot=slot)
    assert b.read_device_status(ws) == 0
    # the appended rows landed, quantised
    d0 = kvp[0].data.cpu().numpy()
    want, _ = ff.fp4_quantize(np32(app))
    for r in range(16):
        s, pos = divmod(int(slot[r]), cap)
        assert np.array_equal(d0[s, pos], want[r])
    wlen = [W, 77]
    for s in range(B):
        kd, ks = ff.fp4_quantize(np32(keys[s]))
        kvals = ff.fp4_dequantize(kd, ks)
        okv = [ff.fp4_quantize(np32(kvs[l][s])) + ("fp4",) for l in range(L)]
        owin = [ff.fp4_quantize(np32(wins[l][s])) for l in range(L)]
        qis = [np32(qi[l][s]) if qi[l] is not None else None for l in range(L)]
        wss = [np32(w[l][s]).astype(np.float64) if w[l] is not None else None for l in range(L)]
        idx_ref, pool_ref, outs_ref = oc.csa2_group_sequence(
            roles, kv_src, idx_src, kvals, n, qis, wss, True, topk, pool_len,
            [np32(q[l][s]) for l in range(L)], okv, owin, wlen[s], TAU)
        # index sets under the R9 contract
        qv0 = oi.indexer_query(qis[0], True)
        s0 = oi.index_scores(qv0, wss[0], kvals)
        e0 = score_eps(qv0, wss[0], kvals)
        gi = [idx_out[l][s].cpu().numpy() for l in range(L)]
        assert check_topk(gi[0], s0, e0, topk, where="full") == 0
        if roles[1] == oc.REINDEX:
            qv1 = oi.indexer_query(qis[1], True)
            s1 = oi.index_scores(qv1, wss[1], kvals)
            e1 = score_eps(qv1, wss[1], kvals)
            assert check_topk(gi[1], s1, e1, topk, candidates=pool_ref, where="reindex") == 0
        for l in range(1, L):
            if roles[l] == oc.REUSE:
                assert np.array_equal(gi[l], gi[idx_src[l]])
        if wiring == "degenerate":
            assert set(gi[1]) == set(gi[0])
        for l in range(L):
            assert np.array_equal(gi[l], idx_ref[l])
            check_attention(out[l][s], lse[l][s], outs_ref[l][0], outs_ref[l][1], H,
                            where="layer %d seq %d" % (l, s))

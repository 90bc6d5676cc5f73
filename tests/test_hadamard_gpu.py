"""Hadamard-rotated FP4 indexer keys (CKV_FMT_FP4H; "DeepSeek-V4 KV Cache
深度分析", §四) through the C ABI against the oracle: the stored bytes of the
append are bit-exact with the oracle's float32 rotation and block quantiser,
and the top-k (the query rotated the same way) matches under the score
contract, on the tensor-core scorer, the CUDA-core scorer (pool rescoring)
and the CSA2 Full pool."""

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from oracle import fp_formats as ff
from oracle import indexer as oi
from tests.helpers import check_topk, ckv, gpu_plane, np32, score_eps

pytestmark = pytest.mark.gpu


def test_fp4h_append_bytes_bit_exact():
    b = ckv()
    x = wl.rms_rows((300, 128), 91, "cuda", spikes=True)
    x[7] = 0
    x[8, :16] = -0.0
    x[9] *= 1000.0
    p = gpu_plane("fp4h", 128, [x], 300)
    d, s = ff.quantize_entries(np32(x), "fp4h")
    assert np.array_equal(p.data.cpu().numpy()[0], d)
    assert np.array_equal(p.scale.cpu().numpy()[0], s)


def _scores(keys, qi, w):
    kd, ks = ff.quantize_entries(np32(keys), "fp4h")
    kv = ff.dequantize_entries(kd, ks, "fp4h")
    qv = oi.indexer_query(np32(qi), True, hadamard=True)
    ww = np32(w).astype(np.float64)
    return oi.index_scores(qv, ww, kv), score_eps(qv, ww, kv)


@pytest.mark.parametrize("HI,n_list,topk", [(64, [9000, 2100], 512), (16, [700], 256), (40, [30000], 512)])
def test_fp4h_index_topk_matches_oracle(HI, n_list, topk):
    b = ckv()
    B = len(n_list)
    keys = [wl.rms_rows((n, 128), 600 + s, "cuda") for s, n in enumerate(n_list)]
    plane = gpu_plane("fp4h", 128, keys, max(n_list) + 4)
    qi = wl.rms_rows((B, HI, 128), 610, "cuda")
    w = wl.head_weights((B, HI), 611, "cuda")
    n_comp = torch.tensor(n_list, dtype=torch.int32, device="cuda")
    dbg = torch.full((B, max(n_list)), float("nan"), device="cuda")
    idx = b.csa_index_topk(plane, n_comp, max(n_list), qi, w, topk, dbg_scores=dbg)
    torch.cuda.synchronize()
    for s in range(B):
        sc, eps = _scores(keys[s], qi[s], w[s])
        got = dbg[s, :n_list[s]].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - sc) <= eps + 1e-30), "score error above the bound"
        assert check_topk(idx[s].cpu().numpy(), sc, eps, topk, where="fp4h seq %d" % s) == 0


def test_fp4h_pool_and_reindex():
    b = ckv()
    n = 12000
    keys = [wl.rms_rows((n, 128), 620 + s, "cuda") for s in range(2)]
    plane = gpu_plane("fp4h", 128, keys, n)
    qi = wl.rms_rows((2, 64, 128), 630, "cuda")
    w = wl.head_weights((2, 64), 631, "cuda")
    n_comp = torch.full((2,), n, dtype=torch.int32, device="cuda")
    idx, pool = b.csa_index_topk(plane, n_comp, n, qi, w, 512, pool_out=2048)
    qi2 = wl.rms_rows((2, 64, 128), 632, "cuda")
    w2 = wl.head_weights((2, 64), 633, "cuda")
    idx2 = b.csa_index_topk(plane, n_comp, n, qi2, w2, 512, pool=pool)
    torch.cuda.synchronize()
    for s in range(2):
        sc, eps = _scores(keys[s], qi[s], w[s])
        assert check_topk(pool[s].cpu().numpy(), sc, eps, 2048, where="pool") == 0
        assert check_topk(idx[s].cpu().numpy(), sc, eps, 512, where="full") == 0
        sc2, eps2 = _scores(keys[s], qi2[s], w2[s])
        p = pool[s].cpu().numpy()
        assert check_topk(idx2[s].cpu().numpy(), sc2, eps2, 512, candidates=p[p >= 0], where="reindex") == 0

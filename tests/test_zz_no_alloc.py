"""The allocation-free index/top-k entry point.

Some callers cannot allocate device memory (serving-engine plug-ins that own
every allocation, embedded runtimes whose memory plan is fixed); for them
ckv_csa_index_topk_static keeps its scratch in a static device array inside
libckv.  These tests call it through the C ABI twice in a row and check that
both calls give exactly what the workspace entry point gives on the same
inputs, and that a device-side range error stays readable through
ckv_read_static_status.  They live in a file pytest collects last."""

import numpy as np

import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from tests.helpers import ckv, gpu_plane

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,HI,n_list,topk,pool_out", [
    ("fp4", 64, [3000, 1500, 700], 512, 0),
    ("fp4", 64, [12000, 9000], 512, 2048),
    ("bf16", 4, [1024], 512, 0),
])
def test_static_scratch_entry_matches_workspace_entry(fmt, HI, n_list, topk, pool_out):
    b = ckv()
    B = len(n_list)
    keys = [wl.rms_rows((n, 128), 4000 + s, "cuda") for s, n in enumerate(n_list)]
    plane = gpu_plane(fmt, 128, keys, max(n_list) + 6)
    qi = wl.rms_rows((B, HI, 128), 4100, "cuda")
    w = wl.head_weights((B, HI), 4200, "cuda")
    n_comp = torch.tensor(n_list, dtype=torch.int32, device="cuda")
    n_max = max(n_list)
    ref = b.csa_index_topk(plane, n_comp, n_max, qi, w, topk, pool_out=pool_out)
    for _ in range(2):
        got = b.csa_index_topk_static(plane, n_comp, n_max, qi, w, topk, pool_out=pool_out)
        torch.cuda.synchronize()
        if pool_out:
            assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        else:
            assert torch.equal(got, ref)


def test_static_scratch_rejects_oversized_calls():
    b = ckv()
    tiny = torch.zeros(256, dtype=torch.uint8, device="cuda")   # never touched: rejected on the host
    plane = b.Plane("fp4", 128, 64, 1 << 20, data=tiny, scale=tiny)
    qi = torch.zeros((64, 64, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((64, 64), device="cuda")
    n_comp = torch.full((64,), 1 << 20, dtype=torch.int32, device="cuda")
    with pytest.raises(b.CkvError) as e:
        b.csa_index_topk_static(plane, n_comp, 1 << 20, qi, w, 2048)
    assert e.value.code == -4


def test_static_scratch_reports_out_of_range_pool_entry():
    """A pool entry at or beyond n_comp is skipped and recorded; the record
    survives the next call's clearing of the counters and reads once."""
    from oracle import fp_formats as ff
    from oracle import indexer as oi
    b = ckv()
    keys = [wl.rms_rows((100, 128), 4300, "cuda")]
    plane = gpu_plane("fp4", 128, keys, 100)
    qi = wl.rms_rows((1, 8, 128), 4301, "cuda")
    w = wl.head_weights((1, 8), 4302, "cuda")
    n_comp = torch.tensor([100], dtype=torch.int32, device="cuda")
    pool = torch.tensor([[5, 7, 250, -1, 9]], dtype=torch.int32, device="cuda")
    assert b.read_static_status() in (0, -6)        # whatever earlier tests left
    idx = b.csa_index_topk_static(plane, n_comp, 100, qi, w, 2, pool=pool)
    good = torch.tensor([[5, 7, 9]], dtype=torch.int32, device="cuda")
    b.csa_index_topk_static(plane, n_comp, 100, qi, w, 2, pool=good)
    assert b.read_static_status() == -6
    assert b.read_static_status() == 0
    kd, ks = ff.fp4_quantize(keys[0].float().cpu().numpy())
    sc = oi.index_scores(oi.indexer_query(qi[0].float().cpu().numpy(), True),
                         w[0].cpu().numpy().astype(np.float64), ff.fp4_dequantize(kd, ks))
    assert list(idx.cpu().numpy()[0]) == list(oi.topk_set(sc, 2, candidates=[5, 7, 9]))

"""The allocation-free index/top-k entry point.

Some callers cannot allocate device memory (code inside a CUDA graph being
captured, serving-engine plug-ins whose memory plan is fixed); for them
ckv_csa_index_topk_static keeps its scratch in a static device array inside
libckv.  This test calls it through the C ABI twice in a row and checks that
both calls give exactly what the workspace entry point gives on the same
inputs.  It lives in a file pytest collects last."""

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

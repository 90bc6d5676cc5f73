"""Failure paths on the GPU, made without faulting it.

* Every spin-wait in the kernels is bounded: ckv_debug_wait_probe runs the
  kernels' wait code on something nothing completes; the wait must give up,
  record CKV_ERR_TIMEOUT in the workspace status word and let the kernel
  return, and the context must stay usable for the next call.
* ckv_csa2_group_decode refuses to be captured into a CUDA graph: on a
  capturing stream it returns CKV_ERR_UNSUPPORTED before enqueueing
  anything (the captured graph is discarded, never replayed)."""

import math
import time

import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from tests.helpers import ckv, gpu_plane

pytestmark = pytest.mark.gpu
TIMEOUT = -5
UNSUPPORTED = -2


def _context_still_usable(b):
    rows = wl.rms_rows((4, 512), 5, "cuda")
    plane = b.Plane("fp4", 512, 1, 4)
    ws = b.new_workspace(256)
    b.kv_append_quant(plane, rows, torch.arange(4, dtype=torch.int64, device="cuda"), ws=ws)
    assert b.read_device_status(ws) == 0
    assert int(plane.data.count_nonzero()) > 0


@pytest.mark.parametrize("mode", [0, 1])
def test_bounded_wait_expires_and_reports_timeout(mode):
    b = ckv()
    ws = b.new_workspace(512)
    t0 = time.perf_counter()
    b.debug_wait_probe(ws, mode, 20000)          # 20 ms
    status = b.read_device_status(ws)            # synchronises
    dt = time.perf_counter() - t0
    assert status == TIMEOUT
    assert 0.015 <= dt < 5.0, dt
    # the status word was cleared by the read, the GPU answers
    assert b.read_device_status(ws) == 0
    _context_still_usable(b)


def test_wait_probe_rejects_bad_arguments():
    b = ckv()
    ws = b.new_workspace(256)
    for mode, lim in [(2, 100), (0, 0), (0, 3000000)]:
        with pytest.raises(b.CkvError) as e:
            b.debug_wait_probe(ws, mode, lim)
        assert e.value.code == -1
    with pytest.raises(b.CkvError) as e:
        b.debug_wait_probe(ws, 1, 100)          # mode 1 needs 512 bytes
    assert e.value.code == -4


def _small_group(b):
    B, n, H, HI, topk, W, L = 1, 600, 64, 64, 64, 128, 3
    keys = gpu_plane("fp4", 128, [wl.rms_rows((n, 128), 61, "cuda")], n)
    kvp = [gpu_plane("fp4", 512, [wl.rms_rows((n, 512), 62 + l, "cuda")], n) for l in range(L)]
    wp = [gpu_plane("fp4", 512, [wl.rms_rows((W, 512), 72 + l, "cuda")], W) for l in range(L)]
    q = [wl.rms_rows((B, H, 512), 81 + l, "cuda") for l in range(L)]
    qi = [wl.rms_rows((B, HI, 128), 91, "cuda"), wl.rms_rows((B, HI, 128), 92, "cuda"), None]
    w = [wl.head_weights((B, HI), 93, "cuda"), wl.head_weights((B, HI), 94, "cuda"), None]
    out = [torch.zeros_like(q[0]) for _ in range(L)]
    g = b.make_group([b.CSA2_FULL, b.CSA2_REINDEX, b.CSA2_REUSE], [0, 0, 2], [0, 0, 0], kvp, wp, keys,
                     q, qi, w, out, pool_len=128)
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    win_len = torch.full((B,), W, dtype=torch.int32, device="cuda")
    ws = b.new_workspace(b.workspace_bytes(b.OP_CSA2, B, H, HI, n, topk, 128))
    return g, n_comp, n, win_len, B, H, HI, topk, ws, out


def test_csa2_group_refuses_stream_capture():
    b = ckv()
    g, n_comp, n, win_len, B, H, HI, topk, ws, out = _small_group(b)
    tau = 1.0 / math.sqrt(512)
    # eager: runs
    b.csa2_group_decode(g, n_comp, n, win_len, B, H, HI, topk, tau, ws=ws)
    assert b.read_device_status(ws) == 0
    assert float(out[0].abs().sum()) > 0
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    code = None
    with torch.cuda.stream(side):
        graph.capture_begin()
        try:
            b.csa2_group_decode(g, n_comp, n, win_len, B, H, HI, topk, tau, ws=ws)
        except b.CkvError as e:
            code = e.code
        finally:
            graph.capture_end()
    del graph                                    # never replayed
    assert code == UNSUPPORTED
    torch.cuda.synchronize()
    # still usable eagerly afterwards
    b.csa2_group_decode(g, n_comp, n, win_len, B, H, HI, topk, tau, ws=ws)
    assert b.read_device_status(ws) == 0

"""The library is reentrant on distinct workspaces: several host threads, each
with its own workspace and stream, call the index/top-k and attention entry
points at once, starting in a fresh process so that the calls' one-time
per-device setup (kernel attributes, occupancy queries, the tensor-map
encoder) runs concurrently too.  Every thread's results must equal, bit for
bit, those of the same calls made one after another."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, threading
import torch
sys.path.insert(0, sys.argv[1])
from compressed_kv_sparse_append_gb300 import binding as b, workloads as wl

B, n, H, HI, W, topk = 4, 3000, 128, 64, 128, 512
dev = "cuda"
keys = b.Plane("fp4", 128, B, n, dev)
kv = b.Plane("mixed", 512, B, n, dev)
win = b.Plane("mixed", 512, B, W, dev)
ws0 = b.new_workspace(256)
for s in range(B):
    base = torch.arange(n, dtype=torch.int64, device=dev) + s * n
    b.kv_append_quant(keys, wl.rms_rows((n, 128), 10 + s, dev), base, ws=ws0)
    b.kv_append_quant(kv, wl.rms_rows((n, 512), 20 + s, dev), base, ws=ws0)
    b.kv_append_quant(win, wl.rms_rows((W, 512), 30 + s, dev),
                      torch.arange(W, dtype=torch.int64, device=dev) + s * W, ws=ws0)
torch.cuda.synchronize()
n_comp = torch.full((B,), n, dtype=torch.int32, device=dev)
win_len = torch.full((B,), W, dtype=torch.int32, device=dev)
T = 4
qi = [wl.rms_rows((B, HI, 128), 100 + t, dev) for t in range(T)]
w = [wl.head_weights((B, HI), 200 + t, dev) for t in range(T)]
q = [wl.rms_rows((B, H, 512), 300 + t, dev) for t in range(T)]
torch.cuda.synchronize()
res = [None] * T
err = []
start = threading.Barrier(T)

def work(t):
    try:
        st = torch.cuda.Stream()
        ws = b.new_workspace(max(b.workspace_bytes(b.OP_INDEX_TOPK, B, H, HI, n, topk, 0),
                                 b.workspace_bytes(b.OP_SPARSE_ATTN, B)))
        torch.cuda.synchronize()
        start.wait()
        with torch.cuda.stream(st):
            idx = b.csa_index_topk(keys, n_comp, n, qi[t], w[t], topk, ws=ws, stream=st)
            out = b.csa_sparse_attn(kv, win, win_len, idx, q[t], 1 / 512 ** 0.5, ws=ws, stream=st)
        st.synchronize()
        if b.read_device_status(ws, st) != 0:
            err.append("device status in thread %d" % t)
        res[t] = (idx.clone(), out.clone())
    except Exception as e:
        err.append("thread %d: %r" % (t, e))

th = [threading.Thread(target=work, args=(t,)) for t in range(T)]
for x in th: x.start()
for x in th: x.join()
assert not err, err
ws = b.new_workspace(max(b.workspace_bytes(b.OP_INDEX_TOPK, B, H, HI, n, topk, 0),
                         b.workspace_bytes(b.OP_SPARSE_ATTN, B)))
for t in range(T):
    idx = b.csa_index_topk(keys, n_comp, n, qi[t], w[t], topk, ws=ws)
    out = b.csa_sparse_attn(kv, win, win_len, idx, q[t], 1 / 512 ** 0.5, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(idx, res[t][0]), "thread %d indices" % t
    assert torch.equal(out.view(torch.int16), res[t][1].view(torch.int16)), "thread %d output" % t
assert b.read_device_status(ws) == 0
print("threads ok")
'''


def test_concurrent_calls_on_distinct_workspaces():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout


def test_index_and_attention_share_one_workspace():
    """index -> attention -> index on one workspace gives the second index
    call the same result as a fresh workspace: the attention's scratch never
    overlaps the index's between-call state (and the other way round)."""
    import torch
    from compressed_kv_sparse_append_gb300 import workloads as wl
    from tests.helpers import ckv
    b = ckv()
    B, n, H, HI, W, topk = 8, 5000, 128, 64, 128, 512
    keys = b.Plane("fp4", 128, B, n)
    kv = b.Plane("mixed", 512, B, n)
    win = b.Plane("mixed", 512, B, W)
    ws0 = b.new_workspace(256)
    for s in range(B):
        base = torch.arange(n, dtype=torch.int64, device="cuda") + s * n
        b.kv_append_quant(keys, wl.rms_rows((n, 128), 40 + s, "cuda"), base, ws=ws0)
        b.kv_append_quant(kv, wl.rms_rows((n, 512), 50 + s, "cuda"), base, ws=ws0)
        b.kv_append_quant(win, wl.rms_rows((W, 512), 60 + s, "cuda"),
                          torch.arange(W, dtype=torch.int64, device="cuda") + s * W, ws=ws0)
    n_comp = torch.full((B,), n, dtype=torch.int32, device="cuda")
    win_len = torch.full((B,), W, dtype=torch.int32, device="cuda")
    shared = b.new_workspace(max(b.workspace_bytes(b.OP_INDEX_TOPK, B, H, HI, n, topk, 0),
                                 b.workspace_bytes(b.OP_SPARSE_ATTN, B),
                                 b.workspace_bytes(b.OP_HCA_ATTN, B)))
    outs = []
    for step in range(3):
        qi = wl.rms_rows((B, HI, 128), 70 + step, "cuda")
        w = wl.head_weights((B, HI), 80 + step, "cuda")
        q = wl.rms_rows((B, H, 512), 90 + step, "cuda")
        idx = b.csa_index_topk(keys, n_comp, n, qi, w, topk, ws=shared)
        out = b.csa_sparse_attn(kv, win, win_len, idx, q, 1 / 512 ** 0.5, ws=shared)
        hout = b.hca_attn(kv, n_comp, n, win, win_len, q, 1 / 512 ** 0.5, ws=shared)
        fresh = b.new_workspace(b.workspace_bytes(b.OP_INDEX_TOPK, B, H, HI, n, topk, 0))
        want = b.csa_index_topk(keys, n_comp, n, qi, w, topk, ws=fresh)
        fresh_a = b.new_workspace(b.workspace_bytes(b.OP_SPARSE_ATTN, B))
        want_o = b.csa_sparse_attn(kv, win, win_len, want, q, 1 / 512 ** 0.5, ws=fresh_a)
        torch.cuda.synchronize()
        assert torch.equal(idx, want), "step %d: indices from the shared workspace" % step
        assert torch.equal(out.view(torch.int16), want_o.view(torch.int16)), "step %d output" % step
        outs.append(hout)
    assert b.read_device_status(shared) == 0

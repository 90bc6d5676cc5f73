"""kv_append_quant (through the C ABI) vs the oracle quantisers: bytes must
be identical."""

import numpy as np
import pytest
import torch

from compressed_kv_sparse_append_gb300 import workloads as wl
from oracle import fp_formats as ff
from tests.helpers import ckv, np32

pytestmark = pytest.mark.gpu


def _rows(n, dim, seed, device="cuda"):
    x = wl.rms_rows((n, dim), seed, device, spikes=True).float()
    # special rows: zeros, negative zeros / tiny negatives, the FP4 extreme
    # (+-2688 and beyond), huge dynamic range within a block
    specials = [lambda r: r.zero_(),
                lambda r: (r.fill_(-0.0), r[::3].fill_(-1e-30)),
                lambda r: r[:16].copy_(torch.tensor([2688.0, -2688.0, 5000.0, 1.0] + [0.5] * 12)),
                lambda r: r.mul_(1e-3),
                lambda r: r[::2].mul_(300.0)]
    for i, f in enumerate(specials[:n]):
        f(x[i])
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("fmt,dim,blk", [("bf16", 512, 448), ("mixed", 512, 448), ("mixed", 512, 64),
                                         ("fp4", 512, 448), ("fp4", 128, 448), ("bf16", 128, 448)])
def test_append_bytes_match_oracle(fmt, dim, blk):
    b = ckv()
    n, B, cap = 77, 3, 40
    src = _rows(n, dim, 11 + dim + blk)
    perm = torch.randperm(B * cap, generator=torch.Generator().manual_seed(5))[:n]
    slot = perm.to(torch.int64)
    slot[7] = -1                                   # skipped row
    plane = b.Plane(fmt, dim, B, cap, nope_block=blk)
    ws = b.new_workspace(256)
    b.kv_append_quant(plane, src.cuda(), slot.cuda(), ws=ws)
    assert b.read_device_status(ws) == 0
    data = plane.data.cpu().numpy().reshape(B * cap, -1)
    want_d, want_s = ff.quantize_entries(np32(src), fmt, blk)
    written = np.zeros(B * cap, bool)
    for r in range(n):
        s = int(slot[r])
        if s < 0:
            continue
        written[s] = True
        assert np.array_equal(data[s], want_d[r]), "row %d data" % r
        if fmt != "bf16":
            sc = plane.scale.cpu().numpy().reshape(B * cap, -1)
            if fmt == "mixed":
                assert np.array_equal(sc[s].view(np.uint32), want_s[r].view(np.uint32)), "row %d scale" % r
            else:
                assert np.array_equal(sc[s], want_s[r]), "row %d scale" % r
    assert not data[~written].any()


def test_append_out_of_range_slot_is_flagged_and_skipped():
    b = ckv()
    plane = b.Plane("fp4", 512, 2, 8)
    src = _rows(3, 512, 3)
    slot = torch.tensor([0, 16, 9], dtype=torch.int64)   # 16 >= 2*8
    ws = b.new_workspace(256)
    b.kv_append_quant(plane, src.cuda(), slot.cuda(), ws=ws)
    assert b.read_device_status(ws) == -6                 # CKV_ERR_DEVICE_BOUNDS
    assert b.read_device_status(ws) == 0                  # cleared
    d = plane.data.cpu().numpy().reshape(16, -1)
    want, _ = ff.fp4_quantize(np32(src))
    assert np.array_equal(d[0], want[0]) and np.array_equal(d[9], want[2])
    assert not np.delete(d, [0, 9], axis=0).any()


def test_append_empty_call():
    b = ckv()
    plane = b.Plane("mixed", 512, 1, 4)
    b.kv_append_quant(plane, torch.empty((0, 512), dtype=torch.bfloat16, device="cuda"),
                      torch.empty((0,), dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert not plane.data.any()


def test_append_multi_matches_single_plane_calls():
    """One launch into three planes (FP4 indexer keys, MIXED and BF16 main KV,
    different row counts, one row skipped) stores what three single calls
    store."""
    b = ckv()
    B, cap = 2, 24
    specs = [("fp4", 128, 448, 9), ("mixed", 512, 64, 13), ("bf16", 512, 448, 4)]
    srcs, slots, multi, single = [], [], [], []
    for i, (fmt, dim, blk, n) in enumerate(specs):
        srcs.append(_rows(n, dim, 300 + i).cuda())
        sl = torch.randperm(B * cap, generator=torch.Generator().manual_seed(40 + i))[:n].to(torch.int64)
        sl[n // 2] = -1
        slots.append(sl.cuda())
        multi.append(b.Plane(fmt, dim, B, cap, nope_block=blk))
        single.append(b.Plane(fmt, dim, B, cap, nope_block=blk))
    ws = b.new_workspace(256)
    b.kv_append_quant_multi(multi, srcs, slots, ws=ws)
    for p, s, sl in zip(single, srcs, slots):
        b.kv_append_quant(p, s, sl, ws=ws)
    assert b.read_device_status(ws) == 0
    for i, (pm, ps) in enumerate(zip(multi, single)):
        assert torch.equal(pm.data, ps.data), "plane %d data" % i
        if pm.scale is not None:
            assert torch.equal(pm.scale.view(torch.uint8), ps.scale.view(torch.uint8)), "plane %d scale" % i
    # and the single calls are pinned to the oracle by test_append_bytes_match_oracle;
    # pin the multi call's FP4 plane directly as well
    want_d, want_s = ff.quantize_entries(np32(srcs[0]), "fp4", 448)
    data = multi[0].data.cpu().numpy().reshape(B * cap, -1)
    for r, s in enumerate(slots[0].cpu().tolist()):
        if s >= 0:
            assert np.array_equal(data[s], want_d[r])

"""Shared test helpers: building cache planes on the GPU (through the C ABI)
and on the oracle side (through oracle.fp_formats) from the same seeded
rows, and the comparison contracts."""

import math

import numpy as np
import torch

from oracle import fp_formats as ff
from oracle import indexer as oi

ATOL = 2e-2      # attention output: max |gpu - oracle|
RTOL = 1e-2      # attention output: per (b, h) ||gpu - oracle|| / ||oracle||
LSE_ATOL = 1e-2


def np32(t):
    return t.detach().to(torch.float32).cpu().numpy()


def ckv():
    import compressed_kv_sparse_append_gb300 as pkg
    from compressed_kv_sparse_append_gb300 import binding
    return binding


def gpu_plane(fmt, dim, rows, cap, nope_block=448, device="cuda"):
    """Plane of len(rows) sequences; rows[b] (bf16 [n_b, dim]) written to
    slots [0, n_b) of sequence b with kv_append_quant."""
    b = ckv()
    B = len(rows)
    plane = b.Plane(fmt, dim, B, cap, device=device, nope_block=nope_block)
    src, slots = [], []
    for s, r in enumerate(rows):
        if r is None or r.shape[0] == 0:
            continue
        src.append(r.to(device))
        slots.append(torch.arange(r.shape[0], dtype=torch.int64, device=device) + s * cap)
    if src:
        ws = b.new_workspace(256, device)
        b.kv_append_quant(plane, torch.cat(src).contiguous(), torch.cat(slots).contiguous(), ws=ws)
        assert b.read_device_status(ws) == 0
    return plane


def oracle_plane(fmt, rows, nope_block=448):
    """Per-sequence (data, scale) numpy planes from the oracle quantiser."""
    out = []
    for r in rows:
        x = np32(r) if r is not None else np.zeros((0, 512), np.float32)
        out.append(ff.quantize_entries(x, fmt, nope_block))
    return out


def score_eps(q_vals, w, key_vals):
    """Per-entry f32 accumulation bound 2^-16 * sum_h w_h sum_i |q_hi k_ji|."""
    a = np.abs(key_vals) @ np.abs(q_vals).T
    return 2.0 ** -16 * (a @ np.abs(w))


def check_topk(got, scores, eps, k, candidates=None, where=""):
    """Exact set equality with the oracle's top-k; a difference is allowed
    only among entries whose oracle scores lie within 2*max(eps) of the
    boundary score, and is reported.  Returns the number of such rows (0 or 1)."""
    want = oi.topk_set(scores, k, candidates)
    got = np.asarray(got, dtype=np.int64)
    g = set(int(v) for v in got if v >= 0)
    w = set(int(v) for v in want if v >= 0)
    assert len(g) == int((got >= 0).sum()), where + ": duplicate indices"
    assert list(got[: len(g)]) == sorted(g), where + ": not ascending / padding in the middle"
    assert all(v == -1 for v in got[len(g):]), where + ": bad padding"
    if g == w:
        return 0
    assert len(g) == len(w), where + ": wrong count"
    sk = np.sort(scores[list(w)])[0]
    e2 = 2 * float(np.max(eps))
    for j in g - w:
        assert scores[j] >= sk - e2, "%s: entry %d (score %r) not near the boundary %r" % (where, j, scores[j], sk)
    for j in w - g:
        assert scores[j] <= sk + e2, "%s: entry %d dropped above the boundary" % (where, j)
    print("near-tie at the top-k boundary (%s): %d entries differ within 2*eps=%g" % (where, len(g - w), e2))
    return 1


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, H, where=""):
    o = np32(o_gpu)[:H]
    diff = np.abs(o - o_ref[:H])
    assert diff.max() <= ATOL, "%s: max abs err %g" % (where, diff.max())
    num = np.linalg.norm(o - o_ref[:H], axis=-1)
    den = np.linalg.norm(o_ref[:H], axis=-1)
    rel = np.where(den > 0, num / np.maximum(den, 1e-30), num)
    assert rel.max() <= RTOL, "%s: rel err %g" % (where, rel.max())
    if lse_gpu is not None:
        lg = lse_gpu.detach().cpu().numpy()[:H].astype(np.float64)
        fin = np.isfinite(lse_ref[:H])
        assert np.array_equal(np.isfinite(lg), fin), where + ": lse finiteness"
        if fin.any():
            assert np.abs(lg[fin] - lse_ref[:H][fin]).max() <= LSE_ATOL, where + ": lse"
    return diff.max(), rel.max()

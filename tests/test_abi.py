"""The C ABI library loads and exports every symbol include/ckv.h declares,
and host-side validation rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "compressed_kv_sparse_append_gb300", "libckv.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from compressed_kv_sparse_append_gb300.build import build
        build()
    return ctypes.CDLL(LIB)


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ckv.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ckv_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    lib.ckv_status_string.restype = ctypes.c_char_p
    for code, name in [(0, b"CKV_OK"), (-1, b"CKV_ERR_INVALID"), (-5, b"CKV_ERR_TIMEOUT"),
                       (-6, b"CKV_ERR_DEVICE_BOUNDS"), (-99, b"CKV_ERR_UNKNOWN")]:
        assert lib.ckv_status_string(code) == name


def test_workspace_sizes(lib):
    f = lib.ckv_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int32] * 7
    assert f(0, 8, 128, 64, 0, 0, 0) == 256
    a = f(1, 4, 128, 64, 262144, 512, 0)
    b = f(1, 8, 128, 64, 262144, 512, 0)
    assert 256 < a < b
    # candidates are sized by the chunking (one slot per entry), not by the
    # pool of a CSA2 Full layer
    assert f(1, 8, 64, 64, 65536, 512, 2048) == f(1, 8, 64, 64, 65536, 512, 0)
    # attention: status word + the shared between-call state (per-sequence
    # index state and 8192-bin histograms, then the attention's merge
    # counters, each 256-byte aligned) + the merge partials of up to 16 CTAs
    # per sequence
    part = 16 * (32 * 128 * 4 + 256) * 4
    zero = 256 + 3 * 8192 * 4 + 256
    assert f(2, 3, 128, 0, 0, 0, 0) == 256 + zero + 3 * part
    assert f(3, 3, 128, 0, 0, 0, 0) == 256 + zero + 3 * part
    # the index/top-k call reserves the same state before its candidates
    assert f(1, 3, 128, 64, 4096, 512, 0) >= 256 + zero
    assert f(4, 8, 64, 64, 65536, 512, 2048) % 256 == 0


def test_host_validation_rejects_before_launch(lib):
    from compressed_kv_sparse_append_gb300.binding import CPlane
    lib.ckv_kv_append_quant.restype = ctypes.c_int32
    # null plane
    assert lib.ckv_kv_append_quant(None, None, None, 0, None, 0, None) == -1
    fake = ctypes.c_void_p(0x10000)
    p = CPlane(2, 512, 448, 1, 8, 0x10000, 0x20000)
    # missing workspace
    assert lib.ckv_kv_append_quant(ctypes.byref(p), fake, fake, 1, None, 0, None) == -4
    # misaligned source
    assert lib.ckv_kv_append_quant(ctypes.byref(p), ctypes.c_void_p(0x10008), fake, 1,
                                   fake, 256, None) == -1
    # unsupported dim / bad format / mixed with an odd scale block
    for bad in (CPlane(2, 256, 448, 1, 8, 0x10000, 0x20000), CPlane(7, 512, 448, 1, 8, 0x10000, 0),
                CPlane(1, 512, 100, 1, 8, 0x10000, 0x20000)):
        assert lib.ckv_kv_append_quant(ctypes.byref(bad), fake, fake, 1, fake, 256, None) in (-1, -2)
    # attention: too many heads, bad workspace size
    kv = CPlane(0, 512, 448, 2, 64, 0x10000, 0)
    lib.ckv_csa_sparse_attn.restype = ctypes.c_int32
    args = [ctypes.byref(kv), ctypes.byref(kv), fake, fake, 2, 512, fake, 256, ctypes.c_float(0.04),
            fake, None, fake, ctypes.c_size_t(256), None]
    assert lib.ckv_csa_sparse_attn(*args) == -2
    args[7] = 128
    args[12] = ctypes.c_size_t(16)
    assert lib.ckv_csa_sparse_attn(*args) == -4


def test_append_multi_host_validation(lib):
    from compressed_kv_sparse_append_gb300.binding import CPlane
    f = lib.ckv_kv_append_quant_multi
    f.restype = ctypes.c_int32
    vp = ctypes.c_void_p
    planes = (CPlane * 2)(CPlane(2, 512, 448, 1, 8, 0x10000, 0x20000),
                          CPlane(2, 128, 448, 1, 8, 0x30000, 0x40000))
    src = (vp * 2)(0x50000, 0x60000)
    slot = (vp * 2)(0x70000, 0x80000)
    n = (ctypes.c_int32 * 2)(1, 1)
    ws = vp(0x90000)
    # no planes, too many planes, null arrays
    assert f(planes, src, slot, n, 0, ws, ctypes.c_size_t(256), None) == -1
    assert f(planes, src, slot, n, 5, ws, ctypes.c_size_t(256), None) == -1
    assert f(None, src, slot, n, 2, ws, ctypes.c_size_t(256), None) == -1
    assert f(planes, None, slot, n, 2, ws, ctypes.c_size_t(256), None) == -1
    # missing workspace
    assert f(planes, src, slot, n, 2, None, ctypes.c_size_t(0), None) == -4
    # a negative row count; a misaligned source of the second plane
    n_bad = (ctypes.c_int32 * 2)(1, -1)
    assert f(planes, src, slot, n_bad, 2, ws, ctypes.c_size_t(256), None) == -1
    src_bad = (vp * 2)(0x50000, 0x60008)
    assert f(planes, src_bad, slot, n, 2, ws, ctypes.c_size_t(256), None) == -1
    # the same plane twice (rows would race)
    same = (CPlane * 2)(planes[0], planes[0])
    assert f(same, src, slot, n, 2, ws, ctypes.c_size_t(256), None) == -1
    # an unsupported dim in the second plane
    odd = (CPlane * 2)(planes[0], CPlane(2, 256, 448, 1, 8, 0x30000, 0x40000))
    assert f(odd, src, slot, n, 2, ws, ctypes.c_size_t(256), None) in (-1, -2)


def _index_args(**over):
    from compressed_kv_sparse_append_gb300.binding import CPlane
    vp = ctypes.c_void_p
    keys = CPlane(2, 128, 448, 2, 64, 0x100000, 0x200000)   # FP4 indexer keys, B = 2, cap 64
    a = dict(keys=keys, n_comp=vp(0x300000), B=2, n_comp_max=64, q=vp(0x400000), w=vp(0x500000),
             HI=64, topk=16, pool=None, pool_len=0, out_idx=vp(0x600000), out_pool=None, pool_out=0,
             dbg=None, ws=vp(0x700000), ws_bytes=ctypes.c_size_t(1 << 30), stream=None)
    a.update(over)
    return [ctypes.byref(a["keys"]), a["n_comp"], a["B"], a["n_comp_max"], a["q"], a["w"], a["HI"],
            a["topk"], a["pool"], a["pool_len"], a["out_idx"], a["out_pool"], a["pool_out"], a["dbg"],
            a["ws"], a["ws_bytes"], a["stream"]]


def test_index_topk_host_validation(lib):
    from compressed_kv_sparse_append_gb300.binding import CPlane
    f = lib.ckv_csa_index_topk
    f.restype = ctypes.c_int32
    vp = ctypes.c_void_p
    assert f(*_index_args(B=0)) == -1                          # no sequences
    assert f(*_index_args(n_comp=None)) == -1                  # null lengths
    assert f(*_index_args(q=vp(0x400008))) == -1               # misaligned query
    assert f(*_index_args(HI=65)) == -2                        # more heads than supported
    assert f(*_index_args(n_comp_max=65)) == -1                # longer than the plane
    assert f(*_index_args(topk=4096)) == -2                    # k above 2048
    assert f(*_index_args(topk=0)) == -2
    # a pool both read and written; a pool smaller than k
    assert f(*_index_args(pool=vp(0x800000), pool_len=32, out_pool=vp(0x900000), pool_out=32)) == -1
    assert f(*_index_args(out_pool=vp(0x900000), pool_out=8)) == -1
    # keys of the wrong width or format
    assert f(*_index_args(keys=CPlane(2, 512, 448, 2, 64, 0x100000, 0x200000))) in (-1, -2)
    assert f(*_index_args(keys=CPlane(1, 128, 448, 2, 64, 0x100000, 0x200000))) in (-1, -2)
    # the workspace: missing, misaligned, too small
    assert f(*_index_args(ws=None)) == -4
    assert f(*_index_args(ws=vp(0x700010))) == -4
    assert f(*_index_args(ws_bytes=ctypes.c_size_t(256))) == -4


def _group(L=6, fmt=2):
    from compressed_kv_sparse_append_gb300.binding import CGroup, CPlane
    g = CGroup()
    g.n_layers = L
    for l in range(L):
        g.role[l] = 0 if l == 0 else (1 if l == 1 else 2)
        g.kv_src[l] = 0
        g.idx_src[l] = 0 if l < 2 else l - 1
        g.kv[l] = CPlane(fmt, 512, 448, 2, 64, 0x1000000 + l * 0x100000, 0x8000000 + l * 0x100000)
        g.win[l] = CPlane(fmt, 512, 448, 2, 16, 0x2000000 + l * 0x100000, 0x9000000 + l * 0x100000)
        g.q[l] = 0x3000000 + l * 0x10000
        g.q_idx[l] = 0x4000000 + l * 0x10000 if l < 2 else None
        g.w[l] = 0x5000000 + l * 0x10000 if l < 2 else None
        g.out[l] = 0x6000000 + l * 0x10000
    g.idx_keys = CPlane(2, 128, 448, 2, 64, 0x7000000, 0x7100000)
    g.pool_len = 32
    return g


def test_csa2_group_host_validation(lib):
    from compressed_kv_sparse_append_gb300.binding import CPlane
    f = lib.ckv_csa2_group_decode
    f.restype = ctypes.c_int32
    vp = ctypes.c_void_p

    def call(g, topk=16, ws_bytes=1 << 30):
        return f(ctypes.byref(g), vp(0xA000000), 64, vp(0xB000000), 2, 64, 64, topk,
                 ctypes.c_float(0.04), None, None, None, 0, vp(0xC000000), ctypes.c_size_t(ws_bytes), None)

    g = _group(); g.n_layers = 0
    assert call(g) == -1
    g = _group(); g.n_layers = 9
    assert call(g) == -1
    g = _group(); g.role[0] = 1                     # the first layer must be a Full layer
    assert call(g) == -1
    g = _group(); g.idx_src[3] = 3                  # Reuse must name an earlier layer
    assert call(g) == -1
    g = _group(); g.kv_src[2] = 6                   # no such layer
    assert call(g) == -1
    g = _group(); g.role[4] = 7                     # no such role
    assert call(g) == -1
    g = _group(); g.pool_len = 8                    # pool smaller than k
    assert call(g) == -1
    g = _group(); g.kv_src[2] = 2; g.kv[2] = CPlane(1, 512, 448, 2, 64, 0x1200000, 0x8200000)
    g.win[2] = CPlane(1, 512, 448, 2, 16, 0x2200000, 0x9200000)
    assert call(g) == -2                            # one launch format across the layers
    assert call(_group(), ws_bytes=256) == -4       # workspace too small


def test_paged_plane_host_validation(lib):
    """Paged planes: whole pages of a multiple of 128 rows, a cap of whole
    pages, dense window rings; FP4H only for 128-d keys."""
    from compressed_kv_sparse_append_gb300.binding import CPlane
    lib.ckv_kv_append_quant.restype = ctypes.c_int32
    fake = ctypes.c_void_p(0x10000)
    bt = 0x50000
    good = CPlane(2, 128, 448, 2, 512, 0x10000, 0x20000, bt, 256, 8)
    assert lib.ckv_kv_append_quant(ctypes.byref(good), fake, fake, 0, fake, 256, None) == 0
    for bad in (CPlane(2, 128, 448, 2, 512, 0x10000, 0x20000, bt, 100, 8),    # page not 128k
                CPlane(2, 128, 448, 2, 500, 0x10000, 0x20000, bt, 256, 8),    # cap not whole pages
                CPlane(2, 128, 448, 2, 512, 0x10000, 0x20000, bt, 256, 0),    # no pages
                CPlane(3, 512, 448, 2, 512, 0x10000, 0x20000, 0, 0, 0)):      # FP4H main KV
        assert lib.ckv_kv_append_quant(ctypes.byref(bad), fake, fake, 1, fake, 256, None) in (-1, -2)
    kv = CPlane(0, 512, 448, 2, 512, 0x10000, 0, bt, 128, 8)
    win = CPlane(0, 512, 448, 2, 128, 0x30000, 0, bt, 128, 2)               # a paged window
    lib.ckv_csa_sparse_attn.restype = ctypes.c_int32
    args = [ctypes.byref(kv), ctypes.byref(win), fake, fake, 2, 512, fake, 128, ctypes.c_float(0.04),
            fake, None, fake, ctypes.c_size_t(1 << 30), None]
    assert lib.ckv_csa_sparse_attn(*args) == -2

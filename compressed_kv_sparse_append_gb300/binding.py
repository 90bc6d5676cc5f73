"""ctypes binding of libckv (argument marshalling only).

Every compute step runs in the library's CUDA kernels; this module turns torch
tensors into device pointers, the current torch stream into a cudaStream_t and
status codes into exceptions.  It raises at import when ``libckv.so`` has not
been built: there is no fallback path.
"""

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libckv.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError("libckv.so is not built (run __graft_entry__.build() or "
                      "python compressed_kv_sparse_append_gb300/build.py)")
lib = ctypes.CDLL(_LIB_PATH)

FMT = {"bf16": 0, "mixed": 1, "fp4": 2, "fp4h": 3}
OP_APPEND, OP_INDEX_TOPK, OP_SPARSE_ATTN, OP_HCA_ATTN, OP_CSA2 = range(5)
CSA2_FULL, CSA2_REINDEX, CSA2_REUSE = 0, 1, 2
MAX_LAYERS = 8

_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class CPlane(ctypes.Structure):
    _fields_ = [("fmt", _i32), ("dim", _i32), ("nope_block", _i32), ("batch", _i32),
                ("cap", _i64), ("data", _vp), ("scale", _vp), ("block_table", _vp),
                ("page_size", _i32), ("n_pages", _i32)]


class CRope(ctypes.Structure):
    _fields_ = [("pos", _vp), ("inv_freq", _vp), ("rotate_q", _i32), ("rotate_out", _i32)]


class Rope:
    """RoPE at the attention's ends (include/ckv.h, ckv_rope): pos [B] int32
    query positions, inv_freq [32] f32 on the device."""

    def __init__(self, pos, inv_freq, rotate_q=True, rotate_out=True):
        self.pos, self.inv_freq = pos, inv_freq
        self.c = CRope(pos.data_ptr(), inv_freq.data_ptr(), int(bool(rotate_q)), int(bool(rotate_out)))


class CGroup(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("role", _i32 * MAX_LAYERS), ("kv_src", _i32 * MAX_LAYERS),
                ("idx_src", _i32 * MAX_LAYERS), ("kv", CPlane * MAX_LAYERS),
                ("win", CPlane * MAX_LAYERS), ("idx_keys", CPlane), ("q", _vp * MAX_LAYERS),
                ("q_idx", _vp * MAX_LAYERS), ("w", _vp * MAX_LAYERS), ("out", _vp * MAX_LAYERS),
                ("lse", _vp * MAX_LAYERS), ("idx_out", _vp * MAX_LAYERS), ("pool_len", _i32),
                ("rope", CRope)]


_P = ctypes.POINTER(CPlane)
lib.ckv_workspace_bytes.restype = _sz
lib.ckv_workspace_bytes.argtypes = [_i32] * 7
lib.ckv_kv_append_quant.restype = _i32
lib.ckv_kv_append_quant.argtypes = [_P, _vp, _vp, _i32, _vp, _sz, _vp]
lib.ckv_kv_append_quant_multi.restype = _i32
lib.ckv_kv_append_quant_multi.argtypes = [_P, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                          ctypes.POINTER(_i32), _i32, _vp, _sz, _vp]
lib.ckv_csa_index_topk.restype = _i32
lib.ckv_csa_index_topk.argtypes = [_P, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp,
                                   _i32, _vp, _vp, _sz, _vp]
lib.ckv_csa_sparse_attn.restype = _i32
lib.ckv_csa_sparse_attn.argtypes = [_P, _P, _vp, _vp, _i32, _i32, _vp, _i32, _f32, _vp, _vp, _vp,
                                    _sz, _vp]
lib.ckv_csa_sparse_attn_rope.restype = _i32
lib.ckv_csa_sparse_attn_rope.argtypes = [_P, _P, _vp, _vp, _i32, _i32, _vp, _i32, _f32, _vp, _vp,
                                         ctypes.POINTER(CRope), _vp, _sz, _vp]
lib.ckv_hca_attn_rope.restype = _i32
lib.ckv_hca_attn_rope.argtypes = [_P, _vp, _i32, _P, _vp, _i32, _vp, _i32, _f32, _vp, _vp,
                                  ctypes.POINTER(CRope), _vp, _sz, _vp]
lib.ckv_hca_attn.restype = _i32
lib.ckv_hca_attn.argtypes = [_P, _vp, _i32, _P, _vp, _i32, _vp, _i32, _f32, _vp, _vp, _vp, _sz, _vp]
lib.ckv_csa2_group_decode.restype = _i32
lib.ckv_csa2_group_decode.argtypes = [ctypes.POINTER(CGroup), _vp, _i32, _vp, _i32, _i32, _i32,
                                      _i32, _f32, _P, _vp, _vp, _i32, _vp, _sz, _vp]
lib.ckv_csa_index_topk_static.restype = _i32
lib.ckv_csa_index_topk_static.argtypes = [_P, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _i32, _vp,
                                          _vp, _i32, _vp, _vp]
lib.ckv_debug_wait_probe.restype = _i32
lib.ckv_debug_wait_probe.argtypes = [_vp, _sz, _i32, ctypes.c_uint32, _vp]
lib.ckv_read_static_status.restype = _i32
lib.ckv_read_static_status.argtypes = [_vp]
lib.ckv_read_device_status.restype = _i32
lib.ckv_read_device_status.argtypes = [_vp, _vp]
lib.ckv_status_string.restype = ctypes.c_char_p
lib.ckv_status_string.argtypes = [_i32]


class CkvError(RuntimeError):
    def __init__(self, code, where):
        super().__init__("%s: %s (%d)" % (where, lib.ckv_status_string(code).decode(), code))
        self.code = code


def _check(code, where):
    if code != 0:
        raise CkvError(code, where)


# Pointers and streams go to ctypes as plain ints (the argtypes convert them):
# a decode step makes a handful of these calls, and on the host each object
# built per argument costs about as much as a kernel launch's own overhead.
def _ptr(t):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def entry_bytes(fmt: str, dim: int) -> int:
    return {"bf16": dim * 2, "mixed": 576, "fp4": dim // 2, "fp4h": dim // 2}[fmt]


def scale_shape(fmt: str, dim: int, nope_block: int = 448):
    if fmt == "mixed":
        return (448 // nope_block,), torch.float32
    if fmt in ("fp4", "fp4h"):
        return (dim // 16,), torch.uint8
    return None, None


class Plane:
    """A cache plane of ``batch`` sequences x ``cap`` entry slots in device
    memory.  Dense: data [batch, cap, entry_bytes] uint8, scale per format.
    Paged (``block_table`` [batch, cap // page_size] int32 on the device):
    data [n_pages * page_size, entry_bytes], scale likewise; entry (b, pos) is
    row block_table[b, pos // page_size] * page_size + pos % page_size.

    The C descriptor is built once and rebuilt whenever a field is
    reassigned; replace ``data`` / ``scale`` by assignment, not by resizing
    the tensors in place (that would move their storage behind the cached
    pointers)."""

    def __init__(self, fmt, dim, batch, cap, device="cuda", nope_block=448, data=None, scale=None,
                 block_table=None, page_size=0, n_pages=0):
        self._c = None
        self.fmt, self.dim, self.batch, self.cap, self.nope_block = fmt, dim, batch, cap, nope_block
        self.block_table, self.page_size, self.n_pages = block_table, page_size, n_pages
        eb = entry_bytes(fmt, dim)
        lead = (n_pages * page_size,) if block_table is not None else (batch, cap)
        self.data = data if data is not None else torch.zeros(lead + (eb,), dtype=torch.uint8,
                                                              device=device)
        shp, dt = scale_shape(fmt, dim, nope_block)
        if scale is not None or shp is None:
            self.scale = scale
        else:
            self.scale = torch.zeros(lead + shp, dtype=dt, device=device)

    def slot(self, b, pos):
        """Row of entry (b, pos) (int64 tensor for tensor pos): the append's slot."""
        if self.block_table is None:
            return pos + b * self.cap
        pg = self.block_table[b][pos // self.page_size].to(torch.int64)
        return pg * self.page_size + pos % self.page_size

    def __setattr__(self, name, value):
        # any change of the plane's fields drops the cached C descriptor
        object.__setattr__(self, name, value)
        if name != "_c":
            object.__setattr__(self, "_c", None)

    def c(self) -> CPlane:
        """The C descriptor (built once, rebuilt after a field is reassigned)."""
        if self._c is None:
            paged = self.block_table is not None
            self._c = CPlane(FMT[self.fmt], self.dim, self.nope_block, self.batch, self.cap,
                             self.data.data_ptr(), None if self.scale is None else self.scale.data_ptr(),
                             self.block_table.data_ptr() if paged else None,
                             self.page_size if paged else 0, self.n_pages if paged else 0)
        return self._c


def workspace_bytes(op, B, H=0, HI=0, n_comp_max=0, topk=0, pool_len=0) -> int:
    return int(lib.ckv_workspace_bytes(op, B, H, HI, n_comp_max, topk, pool_len))


def new_workspace(nbytes, device="cuda"):
    """Zero-filled workspace (256-byte aligned, as torch's allocator returns)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def kv_append_quant(plane: Plane, src, slot, ws=None, stream=None):
    n = 0 if src is None else src.shape[0]
    ws = ws if ws is not None else new_workspace(workspace_bytes(OP_APPEND, 1), plane.data.device)
    c = plane.c()
    _check(lib.ckv_kv_append_quant(c, _ptr(src), _ptr(slot), n, _ptr(ws), ws.numel(),
                                   _stream(stream)), "kv_append_quant")
    return ws


APPEND_MAX_PLANES = 4


def kv_append_quant_multi(planes, srcs, slots, ws=None, stream=None):
    """kv_append_quant into several planes (distinct data) in one launch."""
    k = len(planes)
    if not 1 <= k <= APPEND_MAX_PLANES or len(srcs) != k or len(slots) != k:
        raise ValueError("kv_append_quant_multi: 1..%d planes, one src and slot each" % APPEND_MAX_PLANES)
    ws = ws if ws is not None else new_workspace(workspace_bytes(OP_APPEND, 1), planes[0].data.device)
    cp = (CPlane * k)(*[p.c() for p in planes])
    sp = (_vp * k)(*[_ptr(t) for t in srcs])
    lp = (_vp * k)(*[_ptr(t) for t in slots])
    nn = (_i32 * k)(*[0 if t is None else t.shape[0] for t in srcs])
    _check(lib.ckv_kv_append_quant_multi(cp, sp, lp, nn, k, _ptr(ws), ws.numel(), _stream(stream)),
           "kv_append_quant_multi")
    return ws


def csa_index_topk(keys: Plane, n_comp, n_comp_max, q_idx, w, topk, pool=None, pool_out=0,
                   out_idx=None, out_pool=None, dbg_scores=None, ws=None, stream=None):
    B, HI = q_idx.shape[0], q_idx.shape[1]
    dev = q_idx.device
    if out_idx is None:
        out_idx = torch.empty((B, topk), dtype=torch.int32, device=dev)
    if pool_out and out_pool is None:
        out_pool = torch.empty((B, pool_out), dtype=torch.int32, device=dev)
    if ws is None:
        ws = new_workspace(workspace_bytes(OP_INDEX_TOPK, B, 0, HI, n_comp_max, topk, pool_out), dev)
    pool_len = 0 if pool is None else pool.shape[1]
    c = keys.c()
    _check(lib.ckv_csa_index_topk(c, _ptr(n_comp), B, n_comp_max, _ptr(q_idx), _ptr(w),
                                  HI, topk, _ptr(pool), pool_len, _ptr(out_idx), _ptr(out_pool),
                                  pool_out if out_pool is not None else 0, _ptr(dbg_scores),
                                  _ptr(ws), ws.numel(), _stream(stream)), "csa_index_topk")
    return (out_idx, out_pool) if out_pool is not None else out_idx


def csa_index_topk_static(keys: Plane, n_comp, n_comp_max, q_idx, w, topk, pool=None, pool_out=0,
                          out_idx=None, out_pool=None, dbg_scores=None, stream=None):
    """csa_index_topk with the library's static device scratch instead of a
    caller workspace, for callers that cannot allocate device memory (see
    include/ckv.h); its device status is read with read_static_status."""
    B, HI = q_idx.shape[0], q_idx.shape[1]
    dev = q_idx.device
    if out_idx is None:
        out_idx = torch.empty((B, topk), dtype=torch.int32, device=dev)
    if pool_out and out_pool is None:
        out_pool = torch.empty((B, pool_out), dtype=torch.int32, device=dev)
    pool_len = 0 if pool is None else pool.shape[1]
    c = keys.c()
    _check(lib.ckv_csa_index_topk_static(c, _ptr(n_comp), B, n_comp_max, _ptr(q_idx),
                                         _ptr(w), HI, topk, _ptr(pool), pool_len, _ptr(out_idx),
                                         _ptr(out_pool), pool_out if out_pool is not None else 0,
                                         _ptr(dbg_scores), _stream(stream)), "csa_index_topk_static")
    return (out_idx, out_pool) if out_pool is not None else out_idx


def csa_sparse_attn(kv: Plane, win: Plane, win_len, idx, q, sm_scale, out=None, lse=None, ws=None,
                    stream=None, rope: "Rope" = None):
    B, H = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    ws = ws if ws is not None else new_workspace(workspace_bytes(OP_SPARSE_ATTN, B), q.device)
    ck, cw = kv.c(), win.c()
    if rope is not None:
        _check(lib.ckv_csa_sparse_attn_rope(ck, cw, _ptr(win_len), _ptr(idx), B, idx.shape[1], _ptr(q), H,
                                            sm_scale, _ptr(out), _ptr(lse), ctypes.byref(rope.c), _ptr(ws),
                                            ws.numel(), _stream(stream)), "csa_sparse_attn_rope")
        return out
    _check(lib.ckv_csa_sparse_attn(ck, cw, _ptr(win_len), _ptr(idx), B,
                                   idx.shape[1], _ptr(q), H, sm_scale, _ptr(out), _ptr(lse), _ptr(ws),
                                   ws.numel(), _stream(stream)), "csa_sparse_attn")
    return out


def hca_attn(kv: Plane, n_comp, n_comp_max, win: Plane, win_len, q, sm_scale, out=None, lse=None,
             ws=None, stream=None, rope: "Rope" = None):
    B, H = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    ws = ws if ws is not None else new_workspace(workspace_bytes(OP_HCA_ATTN, B), q.device)
    ck, cw = kv.c(), win.c()
    if rope is not None:
        _check(lib.ckv_hca_attn_rope(ck, _ptr(n_comp), n_comp_max, cw, _ptr(win_len), B, _ptr(q), H, sm_scale,
                                     _ptr(out), _ptr(lse), ctypes.byref(rope.c), _ptr(ws), ws.numel(),
                                     _stream(stream)), "hca_attn_rope")
        return out
    _check(lib.ckv_hca_attn(ck, _ptr(n_comp), n_comp_max, cw,
                            _ptr(win_len), B, _ptr(q), H, sm_scale, _ptr(out), _ptr(lse), _ptr(ws),
                            ws.numel(), _stream(stream)), "hca_attn")
    return out


def make_group(roles, kv_src, idx_src, kv, win, idx_keys, q, q_idx, w, out, lse=None,
               idx_out=None, pool_len=2048, rope: "Rope" = None) -> CGroup:
    g = CGroup()
    L = len(roles)
    g.n_layers = L
    for l in range(L):
        g.role[l], g.kv_src[l], g.idx_src[l] = roles[l], kv_src[l], idx_src[l]
        g.kv[l] = kv[l].c()
        g.win[l] = win[l].c()
        g.q[l] = q[l].data_ptr()
        g.q_idx[l] = q_idx[l].data_ptr() if q_idx[l] is not None else None
        g.w[l] = w[l].data_ptr() if w[l] is not None else None
        g.out[l] = out[l].data_ptr()
        g.lse[l] = lse[l].data_ptr() if lse is not None and lse[l] is not None else None
        g.idx_out[l] = idx_out[l].data_ptr() if idx_out is not None and idx_out[l] is not None else None
    g.idx_keys = idx_keys.c()
    g.pool_len = pool_len
    if rope is not None:
        g.rope = rope.c
        g._rope_keepalive = rope
    return g


def csa2_group_decode(group: CGroup, n_comp, n_comp_max, win_len, B, H, HI, topk, sm_scale,
                      append_dst: Plane = None, append_src=None, append_slot=None, ws=None,
                      stream=None, device="cuda"):
    if ws is None:
        ws = new_workspace(workspace_bytes(OP_CSA2, B, H, HI, n_comp_max, topk, group.pool_len), device)
    n_app = 0 if append_src is None else append_src.shape[0]
    cad = append_dst.c() if append_dst is not None else None
    _check(lib.ckv_csa2_group_decode(ctypes.byref(group), _ptr(n_comp), n_comp_max, _ptr(win_len), B,
                                     H, HI, topk, sm_scale,
                                     ctypes.byref(cad) if cad is not None else None,
                                     _ptr(append_src), _ptr(append_slot), n_app, _ptr(ws), ws.numel(),
                                     _stream(stream)), "csa2_group_decode")
    return ws


def debug_wait_probe(ws, mode, limit_us, stream=None):
    """Runs one of the kernels' bounded waits on something nothing completes
    (mode 0: an mbarrier phase; mode 1: a zero counter in ``ws``); the status
    of ``ws`` then reads CKV_ERR_TIMEOUT (see include/ckv.h)."""
    _check(lib.ckv_debug_wait_probe(_ptr(ws), ws.numel(), mode, limit_us, _stream(stream)),
           "debug_wait_probe")


def read_static_status(stream=None) -> int:
    """Synchronises, returns and clears the sticky device status of the
    static scratch used by csa_index_topk_static (current device)."""
    return int(lib.ckv_read_static_status(_stream(stream)))


def read_device_status(ws, stream=None) -> int:
    """Synchronises, returns and clears the sticky device status of ``ws``."""
    return int(lib.ckv_read_device_status(_ptr(ws), _stream(stream)))

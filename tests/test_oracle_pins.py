"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print (tests/golden/cache_sizes.txt), library conversions (torch's
float8_e4m3fn and bfloat16 casts, scipy's softmax / logsumexp), brute force on
tiny inputs, closed forms, invariants and degenerate cases.
"""

import itertools
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

from oracle import attention, csa2, fp_formats as ff, indexer, sizes
from tests.conftest import load_golden

GOLD = load_golden("cache_sizes.txt")
N1M = 1_048_576


# ----------------------------------------------------------- closed forms --

def test_cache_sizes_bf16_match_printed():
    csa = sizes.per_csa_layer(N1M, "bf16")
    hca = sizes.per_hca_layer(N1M, "bf16")
    tot = sizes.total_bytes(N1M, "bf16")
    assert sizes.fmt_mib(csa) == "%.2f" % GOLD["bf16.csa_layer_mib"]
    assert sizes.fmt_mib(hca) == "%.2f" % GOLD["bf16.hca_layer_mib"]
    assert sizes.fmt_gib(tot) == "%.2f" % GOLD["bf16.total_gib"]
    # exact integers (the formula with the window counted once)
    assert (csa, hca, tot) == (335_675_392, 8_519_680, 10_334_371_840)


def test_cache_sizes_mixed_match_printed():
    csa = sizes.per_csa_layer(N1M, "mixed")
    hca = sizes.per_hca_layer(N1M, "mixed")
    tot = sizes.total_bytes(N1M, "mixed")
    assert sizes.fmt_mib(csa) == "%.2f" % GOLD["mixed.csa_layer_mib"]
    assert sizes.fmt_mib(hca) == "%.2f" % GOLD["mixed.hca_layer_mib"]
    assert sizes.fmt_gib(tot) == "%.2f" % GOLD["mixed.total_gib"]
    assert (csa, hca, tot) == (167_845_888, 4_792_320, 5_183_938_560)


def test_cache_size_components():
    s_kv, s_idx = sizes.entry_bytes("bf16")
    n_c = N1M // 4
    assert n_c * s_kv / sizes.MIB == GOLD["bf16.csa_shared_kv_mib"]
    assert n_c * s_idx / sizes.MIB == GOLD["bf16.csa_indexer_mib"]
    assert (N1M // 128) * s_kv / sizes.MIB == GOLD["bf16.hca_shared_kv_mib"]
    m_kv, m_idx = sizes.entry_bytes("mixed")
    assert (m_kv, m_idx) == (576, 64)
    assert n_c * m_kv / sizes.MIB == GOLD["mixed.csa_comp_kv_mib"]
    assert n_c * m_idx / sizes.MIB == GOLD["mixed.csa_indexer_mib"]
    assert (N1M // 128) * m_kv / sizes.MIB == GOLD["mixed.hca_comp_kv_mib"]


def test_double_counted_window_does_not_match():
    """The appendix listing adds the window twice; that reading misses the
    printed per-layer figures, which confirms the formula's reading."""
    s_kv, s_idx = sizes.entry_bytes("bf16")
    n_c = N1M // 4
    twice = (n_c + 128) * s_kv + n_c * s_idx + 128 * s_kv
    assert sizes.fmt_mib(twice) != "%.2f" % GOLD["bf16.csa_layer_mib"]


def test_cross_model_per_token_arithmetic():
    assert sizes.v3_mla_bytes(N1M) / sizes.GIB == GOLD["v3.total_gib"]
    assert sizes.v32_dsa_bytes(N1M) / sizes.GIB == GOLD["v32.total_gib"]
    assert "%.2f" % float(sizes.v4_pro_no_window_bytes(N1M) / sizes.GIB) == \
        "%.2f" % GOLD["v4pro.nowindow_gib"]
    flash = float(sizes.v4_flash_bytes(N1M) / sizes.GIB)
    assert "%.2f" % flash == "%.2f" % GOLD["v4flash.total_gib"]
    assert "%.1f" % (GOLD["v32.total_gib"] / flash) == "%.1f" % GOLD["v4flash.vs_v32_ratio"]


# ------------------------------------------------------------------ E4M3 --

def _torch_e4m3_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decode_matches_torch():
    ours = ff.e4m3_decode_table()
    ref = _torch_e4m3_table()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert ff.E4M3_MAX == 448.0


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200_000) * rng.choice([1e-3, 1e-1, 1, 10, 100], 200_000),
        np.linspace(-448, 448, 20_001),
        # every midpoint between neighbouring codes (ties to even)
        (ff.e4m3_decode_table()[:126] + ff.e4m3_decode_table()[1:127]) / 2,
        -(ff.e4m3_decode_table()[:126] + ff.e4m3_decode_table()[1:127]) / 2,
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ff.e4m3_encode(x), ref)


def test_e4m3_special_values():
    enc = lambda v: int(ff.e4m3_encode(np.float32(v)))
    assert enc(448) == 0x7E
    assert enc(464) == 0x7E          # midpoint to the would-be 480: even code
    assert enc(480) == 0x7E          # satfinite
    assert enc(1e30) == 0x7E
    assert enc(-1e30) == 0xFE
    assert enc(2.0 ** -10) == 0x00   # half of the smallest subnormal: tie to 0
    assert enc(3 * 2.0 ** -10) == 0x02
    assert enc(-0.0) == 0x80
    assert enc(-2.0 ** -12) == 0x80  # rounds to zero, keeps the sign
    for c in range(256):
        if (c & 0x7F) != 0x7F:
            assert int(ff.e4m3_encode(ff.e4m3_decode(c))) == c


# ------------------------------------------------------------------ E2M1 --

def test_e2m1_values_and_rounding():
    assert list(ff.e2m1_decode_table()[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(ff.e2m1_decode_table()[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             7.0: 6.0, 100.0: 6.0, 0.26: 0.5, 2.51: 3.0, 4.99: 4.0, 5.01: 6.0}
    for x, v in cases.items():
        assert ff.e2m1_decode(ff.e2m1_encode(x)) == v
        assert ff.e2m1_decode(ff.e2m1_encode(-x)) == -v
    for c in range(16):
        assert int(ff.e2m1_encode(ff.e2m1_decode(c))) == c
    assert int(ff.e2m1_encode(-0.1)) == 0x8


def _brute_nearest(r, table):
    """Nearest value of ``table`` by exhaustive search; ties to the even code;
    beyond the largest value, the largest (satfinite)."""
    a = abs(r)
    best = None
    for code, v in enumerate(table):
        d = abs(a - v)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return best[1] | (len(table) if math.copysign(1.0, r) < 0 else 0)


def test_fp4_block_quantiser_brute_force():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 16)) * rng.choice([1e-4, 0.1, 1, 30, 3000], (64, 1)))
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    packed, sc = ff.fp4_quantize(x)
    tab = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for row in range(64):
        amax = float(np.max(np.abs(x[row])))
        s_code = int(ff.e4m3_encode(np.float32(np.float32(amax) / np.float32(6))))
        assert sc[row, 0] == s_code
        s = float(ff.e4m3_decode(s_code))
        for i in range(16):
            c = int((packed[row, i // 2] >> (4 * (i % 2))) & 0xF)
            want = 0 if s == 0 else _brute_nearest(float(np.float32(x[row, i]) / np.float32(s)), tab)
            assert c == want, (row, i)


def test_fp4_max_is_2688():
    """6 x 448 = 2688: a block whose largest element is 2688 gets the top
    scale code and the top value code."""
    x = np.zeros((1, 16), np.float32)
    x[0, 3] = GOLD["fp4.max_representable"]
    x[0, 4] = -GOLD["fp4.max_representable"]
    packed, sc = ff.fp4_quantize(x)
    assert sc[0, 0] == 0x7E and ff.e4m3_decode(0x7E) == 448
    deq = ff.fp4_dequantize(packed, sc)
    assert deq[0, 3] == 2688 and deq[0, 4] == -2688
    assert (packed[0, 1] >> 4) == 0x7 and (packed[0, 2] & 0xF) == 0xF
    # beyond 2688 saturates
    x[0, 3] = 5000
    deq = ff.fp4_dequantize(*ff.fp4_quantize(x))
    assert deq[0, 3] == 2688


def test_fp4_exact_roundtrip_and_nibble_order():
    """Values that are exactly code*scale with amax = 6*scale come back
    bit for bit; the even channel sits in the low nibble."""
    rng = np.random.default_rng(3)
    s_code = rng.integers(0x20, 0x60, size=(50, 2))
    s = ff.e4m3_decode(s_code)
    codes = rng.integers(0, 16, size=(50, 2, 16))
    codes[:, :, 5] = 7                         # amax element = 6 * s
    vals = ff.e2m1_decode(codes) * s[..., None]
    vals = np.where(codes == 8, 0.0, vals).reshape(50, 32).astype(np.float32)
    codes = np.where(codes == 8, 0, codes)     # -0 inputs become +0 here
    packed, sc = ff.fp4_quantize(vals)
    assert np.array_equal(sc, s_code)
    want = (codes[..., 0::2] | (codes[..., 1::2] << 4)).reshape(50, 16)
    assert np.array_equal(packed, want)
    assert np.array_equal(ff.fp4_dequantize(packed, sc), vals)


def test_fp4_error_bound_and_rmsnorm_range():
    """|x - deq| <= half the local E2M1 spacing times s, plus the saturation
    margin of a scale rounded down; an RMS-normalised 512-d vector peaks at
    sqrt(512) ~ 22.6 and stays far below 2688."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((200, 512))
    x = x / np.sqrt((x * x).mean(-1, keepdims=True))
    assert np.abs(x).max() <= math.sqrt(512) + 1e-9
    assert round(math.sqrt(512), 1) == GOLD["rmsnorm.max_abs"]
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    packed, sc = ff.fp4_quantize(x)
    deq = ff.fp4_dequantize(packed, sc)
    s = np.repeat(ff.e4m3_decode(sc), 16, axis=-1)
    r = np.abs(x) / s
    spacing = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    bound = np.where(r <= 6, spacing / 2, r - 6 + 1e-12) * s
    assert np.all(np.abs(x - deq) <= bound + 1e-12)


# --------------------------------------------------------- mixed format ---

def test_mixed_quantiser():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((40, 512))
    x = x / np.sqrt((x * x).mean(-1, keepdims=True))
    xb = torch.from_numpy(x).to(torch.bfloat16)
    x = xb.float().numpy()
    for blk in (448, 64):
        data, s = ff.mixed_quantize(x, blk)
        assert data.shape == (40, 576) and s.shape == (40, 448 // blk)
        # rope bytes are the BF16 bytes, as torch lays them out
        assert np.array_equal(data[:, 448:], xb[:, 448:].contiguous().view(torch.uint8).numpy())
        # scale = fl32(amax / 448); codes = torch's E4M3 cast of fl32(x / s)
        nb = x[:, :448].reshape(40, 448 // blk, blk)
        amax = np.abs(nb).max(-1).astype(np.float32)
        assert np.array_equal(s, amax / np.float32(448))
        r = (nb.astype(np.float32) / s[..., None]).reshape(40, 448)
        ref = torch.from_numpy(r).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(data[:, :448], ref)
        # the largest element of each block maps to +-448
        deq = ff.mixed_dequantize(data, s, blk)
        top = np.abs(ff.e4m3_decode(data[:, :448])).reshape(40, 448 // blk, blk).max(-1)
        assert np.all(top == 448)
        assert np.array_equal(deq[:, 448:], x[:, 448:])
        # |fl32(x/s) - decode(code)| is at most half the local E4M3 step
        # (16 at the top binade [256, 448]); fl32 adds one float32 rounding
        codes_v = ff.e4m3_decode(data[:, :448])
        step = np.where(np.abs(r) < 2.0 ** -6, 2.0 ** -9,
                        2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -6))) - 3))
        assert np.all(np.abs(r - codes_v) <= step / 2)
        assert np.abs(r).max() <= 448 * (1 + 2.0 ** -22)   # fl32 may overshoot; satfinite


def test_zero_block_gives_zero_codes():
    x = np.zeros((2, 512), np.float32)
    data, s = ff.mixed_quantize(x)
    assert not data.any() and not s.any()
    x[1, :16] = -0.0
    packed, sc = ff.fp4_quantize(x)
    assert not packed.any() and not sc.any()


# --------------------------------------------------------------- indexer --

def test_index_scores_worked_example():
    """Hand-computed: q0 = e0, q1 = e1 - e2, w = (0.5, 2).
    k0 = (2, 3, 1, ...) : d = (2, 2)  -> 0.5*2 + 2*2 = 5
    k1 = (-1, 1, 4, ...): d = (-1, -3) -> 0
    k2 = (4, 0, -2, ...): d = (4, 2)  -> 2 + 4 = 6
    k3 = (0, -1, 0, ...): d = (0, -1) -> 0 (ReLU of +-0 is +0)"""
    q = np.zeros((2, 128))
    q[0, 0] = 1
    q[1, 1], q[1, 2] = 1, -1
    keys = np.zeros((4, 128))
    keys[0, :3] = (2, 3, 1)
    keys[1, :3] = (-1, 1, 4)
    keys[2, :3] = (4, 0, -2)
    keys[3, :3] = (0, -1, 0)
    s = indexer.index_scores(q, [0.5, 2.0], keys)
    assert list(s) == [5.0, 0.0, 6.0, 0.0]
    assert not np.signbit(s).any()
    assert list(indexer.topk_set(s, 2)) == [0, 2]
    assert list(indexer.topk_set(s, 3)) == [0, 1, 2]       # tie 1 vs 3 -> lower index
    assert list(indexer.topk_set(s, 6)) == [0, 1, 2, 3, -1, -1]


def test_index_scores_invariants():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((8, 128))
    w = rng.uniform(0, 1, 8)
    k = rng.standard_normal((50, 128))
    s = indexer.index_scores(q, w, k)
    perm = rng.permutation(8)
    assert np.allclose(indexer.index_scores(q[perm], w[perm], k), s, rtol=1e-13, atol=0)
    assert np.allclose(indexer.index_scores(3 * q, w, k), 3 * s, rtol=1e-13, atol=0)
    assert np.allclose(indexer.index_scores(q, 2 * w, k), 2 * s, rtol=1e-13, atol=0)
    # single head, unit weight: ReLU of numpy's dot
    for j in range(50):
        assert indexer.index_scores(q[:1], [1.0], k[j:j + 1])[0] == max(float(np.dot(q[0], k[j])), 0.0)
    # keys in the negative half-space of every head score exactly zero
    assert np.all(indexer.index_scores(np.abs(q), w, -np.abs(k)) == 0)


def test_fp4_indexer_query_is_block_quantised():
    rng = np.random.default_rng(7)
    q = torch.from_numpy(rng.standard_normal((4, 128))).to(torch.bfloat16).float().numpy()
    dq = indexer.indexer_query(q, True)
    assert np.array_equal(dq, ff.fp4_dequantize(*ff.fp4_quantize(q)))
    assert np.array_equal(indexer.indexer_query(q, False), q.astype(np.float64))


def test_topk_brute_force():
    rng = np.random.default_rng(8)
    for trial in range(200):
        n = int(rng.integers(0, 40))
        k = int(rng.integers(1, 20))
        s = rng.integers(0, 6, n).astype(np.float64)  # many exact ties
        if trial % 3 == 0:
            s = rng.standard_normal(n)
        want = sorted(range(n), key=lambda j: (-s[j], j))[:k]
        got = indexer.topk_set(s, k)
        assert sorted(want) == [int(v) for v in got if v >= 0]
        assert list(got[len(want):]) == [-1] * (k - len(want))
        assert all(got[i] < got[i + 1] for i in range(len(want) - 1))


def test_topk_restricted_to_candidates():
    s = np.array([9, 8, 7, 6, 5, 4, 3, 2.0])
    assert list(indexer.topk_set(s, 2, candidates=[7, 3, 5, 1])) == [1, 3]
    assert list(indexer.topk_set(s, 3, candidates=[6, -1])) == [6, -1, -1]


# ------------------------------------------------------------- attention --

def test_attention_matches_scipy_softmax():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((5, 512))
    rows = rng.standard_normal((37, 512))
    tau = 1 / math.sqrt(512)
    o, lse = attention.attend(q, rows, tau)
    z = tau * np.einsum("hd,nd->hn", q, rows)
    a = softmax(z, axis=1)
    assert np.allclose(o, np.einsum("hn,nd->hd", a, rows), rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, logsumexp(z, axis=1), rtol=1e-13, atol=1e-13)


def test_attention_degenerate_cases():
    rng = np.random.default_rng(10)
    tau = 1 / math.sqrt(512)
    q = rng.standard_normal((3, 512))
    e = rng.standard_normal((1, 512))
    o, lse = attention.attend(q, e, tau)                     # one key
    assert np.array_equal(o, np.repeat(e, 3, axis=0))
    assert np.allclose(lse, tau * q @ e[0], rtol=1e-14)
    o, lse = attention.attend(q, np.repeat(e, 9, axis=0), tau)   # identical keys
    assert np.allclose(o, np.repeat(e, 3, axis=0), rtol=1e-14, atol=1e-15)
    assert np.allclose(lse, tau * q @ e[0] + math.log(9), rtol=1e-14)
    rows = rng.standard_normal((11, 512))
    o, lse = attention.attend(np.zeros((2, 512)), rows, tau)    # q = 0 -> mean
    assert np.allclose(o, np.repeat(rows.mean(0, keepdims=True), 2, 0), rtol=1e-13, atol=1e-14)
    assert np.allclose(lse, math.log(11))
    # two keys: logistic weights
    rows = rng.standard_normal((2, 512))
    o, _ = attention.attend(q[:1], rows, tau)
    dz = tau * q[0] @ (rows[0] - rows[1])
    a0 = 1 / (1 + math.exp(-dz))
    assert np.allclose(o[0], a0 * rows[0] + (1 - a0) * rows[1], rtol=1e-12, atol=1e-13)
    # permutation invariance
    rows = rng.standard_normal((20, 512))
    p = rng.permutation(20)
    assert np.allclose(attention.attend(q, rows, tau)[0], attention.attend(q, rows[p], tau)[0],
                       rtol=1e-12, atol=1e-13)
    o, lse = attention.attend(q, np.zeros((0, 512)), tau)      # nothing to attend
    assert not o.any() and np.all(np.isneginf(lse))


def _planes(x, fmt):
    d, s = ff.quantize_entries(x, fmt)
    return d, s


def test_csa_with_all_entries_equals_hca():
    rng = np.random.default_rng(11)
    tau = 1 / math.sqrt(512)
    q = torch.from_numpy(rng.standard_normal((4, 512))).to(torch.bfloat16).float().numpy()
    for fmt in ("bf16", "mixed", "fp4"):
        kv = rng.standard_normal((30, 512))
        kv = torch.from_numpy(kv / np.sqrt((kv ** 2).mean(-1, keepdims=True))).to(torch.bfloat16).float().numpy()
        win = kv[:5] * 0.5
        kd, ks = _planes(kv, fmt)
        wd, ws = _planes(win, fmt)
        oh, lh = attention.hca_attention(q, kd, ks, fmt, 30, wd, ws, 5, tau)
        idx = np.arange(30)[::-1].copy()
        oc, lc = attention.csa_sparse_attention(q, kd, ks, fmt, idx, wd, ws, 5, tau)
        assert np.allclose(oh, oc, rtol=1e-12, atol=1e-13) and np.allclose(lh, lc)
        # no compressed entries: the sliding-window-only layer
        o0, _ = attention.hca_attention(q, kd, ks, fmt, 0, wd, ws, 5, tau)
        ow, _ = attention.attend(q, ff.dequantize_entries(wd, ws, fmt), tau)
        assert np.allclose(o0, ow, rtol=1e-13, atol=1e-14)
        # -1 padding is ignored
        idx = np.array([3, -1, 7, -1])
        o1, _ = attention.csa_sparse_attention(q, kd, ks, fmt, idx, wd, ws, 0, tau)
        o2, _ = attention.attend(q, ff.dequantize_entries(kd[[3, 7]], None if ks is None else ks[[3, 7]], fmt), tau)
        assert np.allclose(o1, o2, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------ CSA2 --

def _csa2_case(rng, n, pool_len, topk):
    tau = 1 / math.sqrt(512)
    keys = torch.from_numpy(rng.standard_normal((n, 128))).to(torch.bfloat16).float().numpy()
    kd, ks = ff.fp4_quantize(keys)
    kvals = ff.fp4_dequantize(kd, ks)
    L = 6
    qi = [torch.from_numpy(rng.standard_normal((8, 128))).to(torch.bfloat16).float().numpy() for _ in range(L)]
    w = [rng.uniform(0, 1, 8) for _ in range(L)]
    q = [torch.from_numpy(rng.standard_normal((4, 512))).to(torch.bfloat16).float().numpy() for _ in range(L)]
    kv, win = [], []
    for l in range(L):
        x = torch.from_numpy(rng.standard_normal((n, 512))).to(torch.bfloat16).float().numpy()
        d, s = ff.fp4_quantize(x)
        kv.append((d, s, "fp4"))
        wx = torch.from_numpy(rng.standard_normal((8, 512))).to(torch.bfloat16).float().numpy()
        win.append(ff.fp4_quantize(wx))
    roles = [csa2.FULL, csa2.REINDEX] + [csa2.REUSE] * 4
    return dict(roles=roles, kv_src=[0, 0, 2, 3, 4, 5], idx_src=[0, 1, 0, 0, 0, 0],
                key_vals=kvals, n_comp=n, q_idx=qi, w=w, idx_fp4=True, topk=topk,
                pool_len=pool_len, q=q, kv=kv, win=win, win_len=8, tau=tau)


def test_csa2_wiring():
    rng = np.random.default_rng(12)
    case = _csa2_case(rng, 300, 64, 16)
    idx, pool, outs = csa2.csa2_group_sequence(**case)
    full_scores = indexer.index_scores(indexer.indexer_query(case["q_idx"][0], True), case["w"][0],
                                       case["key_vals"])
    assert list(idx[0]) == list(indexer.topk_set(full_scores, 16))
    assert set(idx[0]) <= set(pool) and len(set(pool)) == 64
    # Reindex picks only from the pool
    assert set(idx[1]) <= set(pool)
    re_scores = indexer.index_scores(indexer.indexer_query(case["q_idx"][1], True), case["w"][1],
                                     case["key_vals"])
    brute = sorted(pool, key=lambda j: (-re_scores[j], j))[:16]
    assert sorted(brute) == list(idx[1])
    # Reuse layers take layer 0's indices and attend their own KV
    for l in range(2, 6):
        assert list(idx[l]) == list(idx[0])
        d, s, fmt = case["kv"][l]
        wd, ws = case["win"][l]
        o, lse = attention.csa_sparse_attention(case["q"][l], d, s, fmt, idx[0], wd, ws, 8, case["tau"])
        assert np.array_equal(o, outs[l][0]) and np.array_equal(lse, outs[l][1])
    # The Reindex layer attends layer 0's KV
    d, s, fmt = case["kv"][0]
    wd, ws = case["win"][0]
    o, _ = attention.csa_sparse_attention(case["q"][1], d, s, fmt, idx[1], wd, ws, 8, case["tau"])
    assert np.array_equal(o, outs[1][0])


def test_csa2_pool_equal_topk_makes_reindex_a_permutation():
    rng = np.random.default_rng(13)
    case = _csa2_case(rng, 200, 16, 16)
    idx, pool, _ = csa2.csa2_group_sequence(**case)
    assert set(idx[1]) == set(idx[0]) == set(pool)

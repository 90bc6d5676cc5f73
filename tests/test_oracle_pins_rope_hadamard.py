"""Pins of the oracle's RoPE ("DeepSeek-V4 KV Cache 深度分析", §五) and
Hadamard rotation (§四) against what the page and the mathematics fix:
the page's relative-position identity for the output at -i, rotation
algebra (identity, inverse, composition, norms), closed-form angles, the
library's Hadamard matrix, orthonormality, the exact float64 product within
the float32 error bound, and the invariance of unquantised scores."""

import math

import numpy as np
import pytest

from oracle import hadamard as hd
from oracle import indexer as oi
from oracle import rope

RNG = np.random.default_rng(7)
THETA = rope.standard_inv_freq()


def test_rope_identity_at_position_zero_and_nope_untouched():
    x = RNG.standard_normal((5, 512))
    assert np.array_equal(rope.rope_rotate(x, 0, THETA), x)
    y = rope.rope_rotate(x, 123457, THETA)
    assert np.array_equal(y[:, :448], x[:, :448])
    assert not np.allclose(y[:, 448:], x[:, 448:])


def test_rope_closed_form_angle_and_direction():
    # unit real part of pair k: (cos(p theta_k), sin(p theta_k)) at dims
    # (448 + 2k, 449 + 2k): counter-clockwise, real part first
    for k, p in [(0, 1), (0, 3), (5, 1000), (31, 1048575)]:
        x = np.zeros(512)
        x[448 + 2 * k] = 1.0
        y = rope.rope_rotate(x, p, THETA)
        ang = p * float(THETA[k])
        assert abs(y[448 + 2 * k] - math.cos(ang)) < 1e-12
        assert abs(y[449 + 2 * k] - math.sin(ang)) < 1e-12
        # the imaginary unit turns to (-sin, cos)
        x2 = np.zeros(512)
        x2[449 + 2 * k] = 1.0
        y2 = rope.rope_rotate(x2, p, THETA)
        assert abs(y2[448 + 2 * k] + math.sin(ang)) < 1e-12
        assert abs(y2[449 + 2 * k] - math.cos(ang)) < 1e-12


def test_standard_frequencies():
    assert THETA[0] == np.float32(1.0)
    ratio = THETA[1:].astype(np.float64) / THETA[:-1].astype(np.float64)
    assert np.allclose(ratio, 10000.0 ** (-1.0 / 32), rtol=1e-6)


def test_rope_inverse_composition_and_norms():
    x = RNG.standard_normal((3, 512))
    a, b = 77777, -1234
    y = rope.rope_rotate(x, a, THETA)
    assert np.allclose(rope.rope_rotate(y, -a, THETA), x, atol=1e-12)
    assert np.allclose(rope.rope_rotate(y, b, THETA), rope.rope_rotate(x, a + b, THETA), atol=1e-9)
    pn = lambda v: np.hypot(v[..., 448::2], v[..., 449::2])
    assert np.allclose(pn(y), pn(x), atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    # q at position i, entry at position j: the product sees j - i
    q = RNG.standard_normal(512)
    k = RNG.standard_normal(512)
    s1 = rope.rope_rotate(q, 5, THETA) @ rope.rope_rotate(k, 12, THETA)
    s2 = rope.rope_rotate(q, 100005, THETA) @ rope.rope_rotate(k, 100012, THETA)
    assert abs(s1 - s2) < 1e-9 * (abs(s1) + 1)
    s3 = q @ rope.rope_rotate(k, 7, THETA)
    assert abs(s1 - s3) < 1e-9 * (abs(s1) + 1)


def test_output_at_minus_i_turns_absolute_into_relative_positions():
    # the page's identity: R(-i) sum_j a_j R(j) c_j = sum_j a_j R(j - i) c_j
    n, i = 9, 4242
    c = RNG.standard_normal((n, 512))
    pos = RNG.integers(0, 100000, n)
    a = RNG.random(n)
    a /= a.sum()
    stored = np.stack([rope.rope_rotate(c[j], pos[j], THETA) for j in range(n)])
    o, _ = rope.attention_with_rope(lambda qq: (a @ stored, 0.0), np.zeros(512), i, THETA,
                                    rotate_q=False, rotate_out=True)
    want = sum(a[j] * rope.rope_rotate(c[j], pos[j] - i, THETA) for j in range(n))
    assert np.allclose(o, want, atol=1e-12)
    # a wrong sign on the output rotation would miss it
    o_wrong = rope.rope_rotate(a @ stored, i, THETA)
    assert not np.allclose(o_wrong, want, atol=1e-6)


def test_hadamard_matches_library_matrix_and_is_orthonormal():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    h = hd.hadamard_matrix(128)
    assert np.array_equal(h * math.sqrt(128), scipy_linalg.hadamard(128).astype(np.float64))
    assert np.allclose(h @ h.T, np.eye(128), atol=1e-14)
    assert np.allclose(h @ h, np.eye(128), atol=1e-14)     # symmetric: its own inverse


def test_hadamard_f32_butterflies_equal_the_matrix_within_the_f32_bound():
    x = RNG.standard_normal((64, 128)).astype(np.float32)
    x[::7] *= 40.0
    got = hd.hadamard_rotate_f32(x).astype(np.float64)
    exact = hd.hadamard_exact(x)
    # seven rounded stages on partial sums bounded by sum|x|, one rounded scale
    bound = (8 * 2.0 ** -24) * np.abs(x).astype(np.float64).sum(axis=-1, keepdims=True) / math.sqrt(128) \
        + 2.0 ** -24 * np.abs(exact)
    assert np.all(np.abs(got - exact) <= bound)


def test_hadamard_f32_of_unit_vectors_is_exact():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    h = scipy_linalg.hadamard(128).astype(np.float32)
    eye = np.eye(128, dtype=np.float32)
    got = hd.hadamard_rotate_f32(eye)
    assert np.array_equal(got, h * hd.INV_SQRT_N_F32)


def test_rotation_leaves_unquantised_scores_unchanged():
    q = RNG.standard_normal((8, 128))
    k = RNG.standard_normal((50, 128))
    w = RNG.random(8)
    s_plain = oi.index_scores(q, w, k)
    s_rot = oi.index_scores(hd.hadamard_exact(q), w, hd.hadamard_exact(k))
    assert np.allclose(s_plain, s_rot, rtol=1e-12, atol=1e-12)


def test_hadamard_fp4_query_and_keys_round_trip_format():
    from oracle import fp_formats as ff
    x = RNG.standard_normal((10, 128)).astype(np.float32)
    d, s = ff.quantize_entries(x, "fp4h")
    d2, s2 = ff.fp4_quantize(hd.hadamard_rotate_f32(x))
    assert np.array_equal(d, d2) and np.array_equal(s, s2)
    v = ff.dequantize_entries(d, s, "fp4h")
    # the dequantised rotated keys are within half an E2M1 step (times the
    # block scale) of the rotated values: steps 0.5 below 2, 1 below 4, 2 up to 6
    rot = hd.hadamard_rotate_f32(x).astype(np.float64)
    sc = ff.e4m3_decode(s).repeat(16, axis=-1)
    r = np.abs(rot) / sc
    half_step = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0)) * sc
    assert np.all(np.abs(v - rot) <= half_step * (1 + 1e-6) + 1e-12)
    qv = oi.indexer_query(x[:2], True, hadamard=True)
    assert np.array_equal(qv, ff.fp4_dequantize(*ff.fp4_quantize(hd.hadamard_rotate_f32(x[:2]))))


def test_paged_layout_round_trip():
    """A paged plane holds the dense plane's entries: every logical entry
    comes back from its page, with an identity table the paged array is the
    dense one, and distinct table entries never alias."""
    from oracle import paged
    B, cap, ps, n_pages = 3, 512, 128, 16
    dense = RNG.integers(0, 256, (B, cap, 7)).astype(np.uint8)
    ident = np.arange(B * cap // ps).reshape(B, cap // ps)
    assert np.array_equal(paged.paged_from_dense(dense, ident, ps, B * cap // ps), dense.reshape(B * cap, 7))
    table = RNG.permutation(n_pages)[:B * cap // ps].reshape(B, cap // ps)
    pg = paged.paged_from_dense(dense, table, ps, n_pages)
    for b in range(B):
        assert np.array_equal(paged.logical_rows(pg, table, ps, b, cap), dense[b])
    rows = np.concatenate([paged.row_of(table, ps, b, np.arange(cap)) for b in range(B)])
    assert len(set(rows.tolist())) == B * cap

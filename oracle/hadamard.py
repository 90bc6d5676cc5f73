"""Hadamard rotation of the 128-d indexer vectors before FP4 (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"DeepSeek-V4 KV Cache 深度分析", §四 (indexer): the indexer's FP4 quantisation
is a Hadamard rotation followed by ``fp4_act_quant`` over all 128 dims.  An
orthogonal rotation applied to both the query and the key leaves every
unquantised product q . k unchanged; it spreads each vector's energy over
all channels before the block quantiser sees it.

Readings (the pages name the steps only):
  * the rotation is the Sylvester-ordered Hadamard matrix of order 128,
    normalised by 1/sqrt(128) so that it is orthonormal (H H^T = I);
    x -> x H (H is symmetric);
  * the quantised bytes must match bit for bit, and the pages fix no
    precision, so the rotated values are the kernel's: float32 butterflies
    of the fast Walsh-Hadamard transform in its canonical order (stage
    h = 1, 2, 4, ..., 64; pair (j, j + h) for every j with bit h clear
    becomes (a + b, a - b)), then one float32 multiplication by
    fl32(1/sqrt(128)); the float64 product x H is the exact value they
    approximate (pinned within the float32 error bound);
  * the query is rotated the same way before its own FP4 quantisation; both
    are then the E2M1 + E4M3/16 block quantiser of ``fp_formats``.
"""

import numpy as np

from .fp_formats import fp4_quantize

N = 128
INV_SQRT_N_F32 = np.float32(1.0 / np.sqrt(N))


def hadamard_matrix(n: int = N) -> np.ndarray:
    """Sylvester construction, normalised: H_1 = [1], H_2m = [[H, H],
    [H, -H]], divided by sqrt(n).  float64 [n, n]."""
    assert n > 0 and (n & (n - 1)) == 0
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(n)


def hadamard_exact(x) -> np.ndarray:
    """x [..., 128] -> x H in float64."""
    return np.asarray(x, dtype=np.float64) @ hadamard_matrix(np.asarray(x).shape[-1])


def hadamard_rotate_f32(x) -> np.ndarray:
    """The rotation as the kernels compute it: float32 butterflies in the
    canonical order, then the float32 scale.  x [..., 128] -> float32."""
    v = np.array(x, dtype=np.float32, copy=True)
    n = v.shape[-1]
    h = 1
    while h < n:
        v = v.reshape(v.shape[:-1] + (n // (2 * h), 2, h))
        a = v[..., 0, :].copy()
        b = v[..., 1, :].copy()
        v[..., 0, :] = a + b          # float32 sums
        v[..., 1, :] = a - b
        v = v.reshape(v.shape[:-3] + (n,))
        h *= 2
    return (v * INV_SQRT_N_F32).astype(np.float32)


def fp4_quantize_hadamard(x):
    """FP4 codes and scales of the Hadamard-rotated vectors (same packing as
    ``fp_formats.fp4_quantize``)."""
    return fp4_quantize(hadamard_rotate_f32(x))

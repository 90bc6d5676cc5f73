"""RoPE at the two ends of the decode attention (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"DeepSeek-V4 KV Cache 深度分析", §五 (RoPE, three sites): rotary position
embedding acts on the last 64 dims of (1) the query, (2) each compressed KV
entry and (3) the core attention output, the output at position -i.  The
page's reason: each entry is both key and value and carries the absolute
position of its own rotation, so the output sum_j a_j R(j) c_j carries
absolute positions; rotating it by -i turns every term into R(j - i) c_j, a
position relative to the query.  Site (2) happens when an entry is written
(entries reach the cache already rotated); sites (1) and (3) belong to the
attention step and are computed here.

Readings (the pages give no formula for the rotation itself):
  * the 64 RoPE dims form 32 pairs of adjacent dims (2k, 2k + 1) of the
    rope part, each pair one complex number (real part first), as the
    page's ``freqs_cis`` (complex frequencies) suggests;
  * pair k turns by the angle pos * theta_k; the frequencies theta_k are
    an input (the model's own table, e.g. base^(-2k/64), possibly scaled for
    long context); ``standard_inv_freq`` gives the plain base-10000 one;
  * i is the query token's position; the query turns by +i and the output
    by -i; the angle is pos * theta_k with theta_k taken as given (float32
    values, exact in float64).

Everything in float64.
"""

import numpy as np

ROPE_DIM = 64
N_PAIRS = ROPE_DIM // 2


def standard_inv_freq(base: float = 10000.0) -> np.ndarray:
    """theta_k = base^(-2k / 64) for k = 0..31, as float32."""
    k = np.arange(N_PAIRS, dtype=np.float64)
    return (base ** (-2.0 * k / ROPE_DIM)).astype(np.float32)


def rope_rotate(x, pos, inv_freq) -> np.ndarray:
    """x [..., D] -> float64 copy whose last 64 dims are turned by the angle
    pos * theta_k, pair k = dims (D - 64 + 2k, D - 64 + 2k + 1) as a complex
    number (real, imaginary).  pos: a scalar or an array broadcasting against
    x's leading dims."""
    x = np.array(x, dtype=np.float64, copy=True)
    D = x.shape[-1]
    theta = np.asarray(inv_freq, dtype=np.float32).astype(np.float64)
    assert theta.shape == (N_PAIRS,)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta          # [..., 32]
    c, s = np.cos(ang), np.sin(ang)
    re = x[..., D - ROPE_DIM::2].copy()
    im = x[..., D - ROPE_DIM + 1::2].copy()
    x[..., D - ROPE_DIM::2] = re * c - im * s
    x[..., D - ROPE_DIM + 1::2] = re * s + im * c
    return x


def attention_with_rope(attend_fn, q, pos, inv_freq, rotate_q: bool, rotate_out: bool):
    """Site (1), the attention, site (3): q [H, D] turned by +pos when
    rotate_q; attend_fn(q) -> (o, lse); o turned by -pos when rotate_out.
    The lse is that of the attention (the rotation of o does not change it)."""
    qq = rope_rotate(q, pos, inv_freq) if rotate_q else np.asarray(q, dtype=np.float64)
    o, lse = attend_fn(qq)
    if rotate_out:
        o = rope_rotate(o, -np.float64(pos), inv_freq)
    return o, lse

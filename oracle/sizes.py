"""KV-cache size closed forms (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"DeepSeek-V4 KV Cache 深度分析", §七 (general formula) gives, for a context
of N tokens, a sliding window of w entries and per-entry byte sizes S_kv
(main KV) and S_idx (indexer key):

    PerCSA = (N/4 + w) * S_kv + (N/4) * S_idx
    PerHCA = (N/128 + w) * S_kv
    Total  = N_CSA * PerCSA + N_HCA * PerHCA

N/ratio is the integer count of compressed entries.  The entry sizes follow
from §六's precision table (bytes per element of each part of an entry) and
§二's entry layout (a 512-d latent whose last 64 dims carry RoPE; the
indexer key of §四 is 128-d).  The layer counts are §一's (V4-Pro: 30 CSA and
31 HCA layers), the ratios and window §三's.

Reading: the window is counted once.  The page's appendix calculator adds it
a second time, but the per-layer and GiB figures it prints equal the §七
formula with a single window, so those printed figures, not the listed
code, are what this module reproduces.

Also the per-token arithmetic of "DeepSeek V4 의 정확한 KV 캐시 사용량 분석"
(V3 MLA, V3.2 with its indexer, V4-Pro without window, V4-Flash with two
sliding-window layers).
"""

from collections import namedtuple
from fractions import Fraction

MIB = 1 << 20
GIB = 1 << 30

# §二 / §四: shape of one compressed entry and one indexer key.
Geometry = namedtuple("Geometry", "latent rope index")
ENTRY = Geometry(latent=512, rope=64, index=128)

# §三: compression ratios and window; §一: V4-Pro layer counts.
Model = namedtuple("Model", "csa_ratio hca_ratio window n_csa n_hca")
V4_PRO = Model(csa_ratio=4, hca_ratio=128, window=128, n_csa=30, n_hca=31)

# §六: bytes per element of each part of a cache entry, per deployment.
#   "bf16"  : everything BF16.
#   "mixed" : RoPE dims BF16, the other latent dims FP8, indexer keys FP4.
# Scale bytes are not part of the page's entry sizes.
BYTES_PER_ELEMENT = {
    "bf16": {"nope": Fraction(2), "rope": Fraction(2), "index": Fraction(2)},
    "mixed": {"nope": Fraction(1), "rope": Fraction(2), "index": Fraction(1, 2)},
}


def entry_bytes(precision: str):
    """(S_kv, S_idx): bytes of one main-KV entry and one indexer key."""
    b = BYTES_PER_ELEMENT[precision]
    nope = ENTRY.latent - ENTRY.rope
    s_kv = nope * b["nope"] + ENTRY.rope * b["rope"]
    s_idx = ENTRY.index * b["index"]
    return int(s_kv), int(s_idx)


def _layer(n_tokens: int, ratio: int, window: int, s_kv: int, s_idx: int) -> int:
    """One layer of the §七 formula: compressed entries and window at S_kv,
    plus one indexer key per compressed entry (S_idx = 0 without indexer)."""
    n_c = n_tokens // ratio
    return (n_c + window) * s_kv + n_c * s_idx


def per_csa_layer(n_tokens: int, precision: str, window: int = V4_PRO.window) -> int:
    s_kv, s_idx = entry_bytes(precision)
    return _layer(n_tokens, V4_PRO.csa_ratio, window, s_kv, s_idx)


def per_hca_layer(n_tokens: int, precision: str, window: int = V4_PRO.window) -> int:
    s_kv, _ = entry_bytes(precision)
    return _layer(n_tokens, V4_PRO.hca_ratio, window, s_kv, 0)


def total_bytes(n_tokens: int, precision: str, n_csa: int = V4_PRO.n_csa,
                n_hca: int = V4_PRO.n_hca) -> int:
    return n_csa * per_csa_layer(n_tokens, precision) + n_hca * per_hca_layer(n_tokens, precision)


def fmt_mib(b: int) -> str:
    """'%.2f' of the exact binary value b / 2**20 (round half to even on the
    exact value, as Python's float formatting of an exact dyadic does)."""
    return "%.2f" % (b / MIB)


def fmt_gib(b: int) -> str:
    return "%.2f" % (b / GIB)


# --- per-token arithmetic of the V3 / V3.2 / V4 comparison page ----------

def v3_mla_bytes(n_tokens: int, n_layers: int = 61) -> int:
    """MLA caches the 512-d latent and the 64-d RoPE key in BF16 per token
    and layer."""
    return (ENTRY.latent + ENTRY.rope) * 2 * n_layers * n_tokens


def v32_dsa_bytes(n_tokens: int, n_layers: int = 61) -> int:
    """V3.2 also caches the 128-d indexer key per token (BF16)."""
    return (ENTRY.latent + ENTRY.rope + ENTRY.index) * 2 * n_layers * n_tokens


def v4_pro_no_window_bytes(n_tokens: int) -> Fraction:
    """Per token: CSA keeps (latent + indexer key) in BF16 for every 4
    tokens, HCA the latent for every 128; 30 + 31 layers, window omitted."""
    csa = Fraction((ENTRY.latent + ENTRY.index) * 2, V4_PRO.csa_ratio)
    hca = Fraction(ENTRY.latent * 2, V4_PRO.hca_ratio)
    return (csa * V4_PRO.n_csa + hca * V4_PRO.n_hca) * n_tokens


def v4_flash_bytes(n_tokens: int) -> Fraction:
    """V4-Flash: 21 CSA + 20 HCA layers, plus two sliding-window layers
    whose padded per-layer cache is 2*1*128*2*(128+256) = 196608 bytes."""
    csa = Fraction((ENTRY.latent + ENTRY.index) * 2, V4_PRO.csa_ratio)
    hca = Fraction(ENTRY.latent * 2, V4_PRO.hca_ratio)
    swa = 2 * 1 * 128 * 2 * (128 + 256)
    return (csa * 21 + hca * 20) * n_tokens + 2 * swa

"""KV-cache size closed forms (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows "DeepSeek-V4 KV Cache 深度分析", §七 (general formula): with N
tokens, window w and per-entry byte sizes S_kv / S_idx,

    PerCSA = (N/4 + w) * S_kv + (N/4) * S_idx
    PerHCA = (N/128 + w) * S_kv
    Total  = N_CSA * PerCSA + N_HCA * PerHCA,

with N/ratio taken as the integer number of compressed entries.  The entry
sizes are those of §六's precision table (BF16: S_kv = 512*2, S_idx = 128*2;
mixed: S_kv = 448*1 + 64*2, S_idx = 128/2) and the layer counts those of §一
(30 CSA + 31 HCA for V4-Pro).

The page's appendix calculator adds the window a second time (its
``csa_compressed`` already includes it); its printed per-layer and GiB figures
match the §七 formula with the window counted once, which is the reading used
here.

Also the per-token byte arithmetic of "DeepSeek V4 의 정확한 KV 캐시 사용량
분석" (V3 MLA, V3.2 with the 128-byte indexer, V4-Pro without window, V4-Flash
with two sliding-window layers).
"""

from fractions import Fraction

HEAD_DIM = 512
ROPE_DIM = 64
NOPE_DIM = HEAD_DIM - ROPE_DIM
INDEX_DIM = 128
WINDOW = 128
CSA_RATIO = 4
HCA_RATIO = 128
N_CSA = 30
N_HCA = 31

MIB = 1 << 20
GIB = 1 << 30


def entry_bytes(precision: str):
    """(S_kv, S_idx) in bytes per compressed entry, scales excluded."""
    if precision == "bf16":
        return HEAD_DIM * 2, INDEX_DIM * 2
    if precision == "mixed":
        return NOPE_DIM * 1 + ROPE_DIM * 2, INDEX_DIM // 2
    raise ValueError(precision)


def per_csa_layer(n_tokens: int, precision: str, window: int = WINDOW) -> int:
    s_kv, s_idx = entry_bytes(precision)
    n_c = n_tokens // CSA_RATIO
    return (n_c + window) * s_kv + n_c * s_idx


def per_hca_layer(n_tokens: int, precision: str, window: int = WINDOW) -> int:
    s_kv, _ = entry_bytes(precision)
    return (n_tokens // HCA_RATIO + window) * s_kv


def total_bytes(n_tokens: int, precision: str, n_csa: int = N_CSA, n_hca: int = N_HCA) -> int:
    return n_csa * per_csa_layer(n_tokens, precision) + n_hca * per_hca_layer(n_tokens, precision)


def fmt_mib(b: int) -> str:
    """'%.2f' of the exact binary value b / 2**20 (round half to even on the
    exact value, as Python's float formatting of an exact dyadic does)."""
    return "%.2f" % (b / MIB)


def fmt_gib(b: int) -> str:
    return "%.2f" % (b / GIB)


# --- per-token arithmetic of the V3 / V3.2 / V4 comparison page ----------

def v3_mla_bytes(n_tokens: int, n_layers: int = 61) -> int:
    """(kv_lora_rank 512 + rope 64) * 2 bytes per token per layer."""
    return (512 + 64) * 2 * n_layers * n_tokens


def v32_dsa_bytes(n_tokens: int, n_layers: int = 61) -> int:
    """V3.2 adds the 128-dim indexer: (512 + 64 + 128) * 2 bytes."""
    return (512 + 64 + 128) * 2 * n_layers * n_tokens


def v4_pro_no_window_bytes(n_tokens: int) -> Fraction:
    """CSA (512+128)*2/4 = 320 B and HCA 512*2/128 = 8 B per token per
    layer, 30 + 31 layers, window omitted."""
    csa = Fraction((512 + 128) * 2, 4)
    hca = Fraction(512 * 2, 128)
    return (csa * 30 + hca * 31) * n_tokens


def v4_flash_bytes(n_tokens: int) -> Fraction:
    """21 CSA + 20 HCA layers plus two sliding-window layers whose padded
    per-layer cache is 2*1*128*2*(128+256) = 196608 bytes."""
    csa = Fraction((512 + 128) * 2, 4)
    hca = Fraction(512 * 2, 128)
    swa = 2 * 1 * 128 * 2 * (128 + 256)
    return (csa * 21 + hca * 20) * n_tokens + 2 * swa

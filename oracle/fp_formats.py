"""Number formats and block quantisers of the compressed KV cache (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Formats, from the pages:
  * mixed storage of a 512-d entry: the 448 "nope" dims in FP8, the 64 RoPE
    dims kept in BF16 -- "DeepSeek-V4 KV Cache 深度分析", §二 (KV entry
    figure) and §六 (precision table); the quantiser call ``act_quant`` on the
    first 448 dims is quoted in §二's code evidence.
  * FP4 E2M1 values with one E4M3 scale per 16 channels and no global scale --
    "V4.1-Flash 공개", 핵심 내용 (third paragraph); "KV cache 890 bajtów na
    token", "Trzy mechanizmy" (third mechanism).  The 4-bit indexer keys of
    §四 use the same block format here.

Everything is computed in float64 from the format definitions (OCP FP8 E4M3
"fn": bias 7, no infinities, S.1111.111 = NaN, max 448; E2M1: bias 1, values
±{0, .5, 1, 1.5, 2, 3, 4, 6}).  Rounding is round-to-nearest-even on the exact
value with saturation to the largest finite magnitude ("satfinite").

Readings (where the pages are silent): the quotient x / s and amax / 6,
amax / 448 are formed in IEEE float32 (the arithmetic type of the quantiser);
codes carry the sign of x (negative values that round to zero give the
negative-zero code); a block whose scale is zero stores all-zero codes; the
even channel of a pair sits in the low nibble of an FP4 byte; FP8 scales of the
mixed format are float32, one per block of ``nope_block`` channels (448 = one
per entry).
"""

import numpy as np

# ---------------------------------------------------------------- E4M3 ----


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 E4M3 codes, from the bit-field definition."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)  # subnormal
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3 = e4m3_decode_table()
_E4M3_POS = _E4M3[:127]          # codes 0x00..0x7E, strictly increasing
E4M3_MAX = float(_E4M3[0x7E])    # 448


def _rne_encode(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of the increasing ``table`` to each
    non-negative magnitude, ties to the even index, saturating at the top."""
    mag = np.asarray(mag, dtype=np.float64)
    top = len(table) - 1
    hi = np.searchsorted(table, mag, side="left")
    hi = np.clip(hi, 0, top)
    lo = np.clip(hi - 1, 0, top)
    d_lo = mag - table[lo]
    d_hi = table[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= table[top], top, idx)      # satfinite
    idx = np.where(mag <= 0.0, 0, idx)
    return idx.astype(np.int64)


def _negative(x: np.ndarray) -> np.ndarray:
    return np.signbit(np.asarray(x, dtype=np.float64))


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even, satfinite E4M3 code (uint8) of each value."""
    x = np.asarray(x, dtype=np.float64)
    code = _rne_encode(np.abs(x), _E4M3_POS)
    code = np.where(_negative(x), code | 0x80, code)
    return code.astype(np.uint8)


def e4m3_decode(code) -> np.ndarray:
    return _E4M3[np.asarray(code, dtype=np.int64)]


# ---------------------------------------------------------------- E2M1 ----

def e2m1_decode_table() -> np.ndarray:
    """Value of each of the 16 E2M1 codes (1 sign, 2 exponent bits with bias
    1, 1 mantissa bit; exponent field 0 is subnormal)."""
    vals = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        e = (code >> 1) & 0x3
        m = code & 0x1
        if e == 0:
            vals[code] = sign * (m / 2.0) * 2.0 ** (1 - 1)
        else:
            vals[code] = sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return vals


_E2M1 = e2m1_decode_table()
_E2M1_POS = _E2M1[:8]            # 0, .5, 1, 1.5, 2, 3, 4, 6
E2M1_MAX = float(_E2M1[7])       # 6


def e2m1_encode(x) -> np.ndarray:
    """Round-to-nearest-even, saturating E2M1 code (0..15) of each value."""
    x = np.asarray(x, dtype=np.float64)
    code = _rne_encode(np.abs(x), _E2M1_POS)
    code = np.where(_negative(x), code | 0x8, code)
    return code.astype(np.uint8)


def e2m1_decode(code) -> np.ndarray:
    return _E2M1[np.asarray(code, dtype=np.int64)]


# ---------------------------------------------------------------- BF16 ----

def bf16_bytes(x) -> np.ndarray:
    """Little-endian bytes of values that are exactly representable in BF16
    (the inputs of the cache are BF16; no rounding happens here)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = f.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("bf16_bytes: value not exactly representable in BF16")
    hi = (bits >> 16).astype(np.uint16)
    return hi.view(np.uint8).reshape(f.shape[:-1] + (f.shape[-1] * 2,))


def bf16_from_bytes(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint8))
    hi = b.view(np.uint16).astype(np.uint32) << 16
    return hi.view(np.float32).astype(np.float64)


# ------------------------------------------------ FP4 block quantiser ----

FP4_BLOCK = 16


def fp4_quantize(x):
    """E2M1 codes with one E4M3 scale per 16 channels.

    For each block of 16 channels: amax = max |x|; the scale code is
    E4M3(fl32(amax / 6)) (6 = largest E2M1 magnitude, so the block's largest
    element lands on the top code); s is its value; the codes are
    E2M1(fl32(x / s)), or all zero when s == 0.

    Returns (packed bytes [..., D/2] uint8, scale codes [..., D/16] uint8).
    """
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    assert D % FP4_BLOCK == 0
    xb = x.reshape(x.shape[:-1] + (D // FP4_BLOCK, FP4_BLOCK))
    amax = np.abs(xb).max(axis=-1)
    s_code = e4m3_encode(np.float32(amax) / np.float32(6.0))
    s = e4m3_decode(s_code)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = xb / s.astype(np.float32)[..., None]          # float32 quotient
    codes = e2m1_encode(r)
    codes = np.where((s > 0)[..., None], codes, 0).astype(np.uint8)
    codes = codes.reshape(x.shape[:-1] + (D,))
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, s_code


def fp4_dequantize(packed, s_code) -> np.ndarray:
    """float64 values of packed E2M1 codes times their block's E4M3 scale."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0xF
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (packed.shape[-1] * 2,))
    v = e2m1_decode(codes)
    s = e4m3_decode(s_code)
    D = v.shape[-1]
    v = v.reshape(v.shape[:-1] + (D // FP4_BLOCK, FP4_BLOCK)) * s[..., None]
    return v.reshape(v.shape[:-2] + (D,))


# --------------------------------- mixed FP8-nope / BF16-rope entries ----

MAIN_DIM = 512
ROPE_DIM = 64
NOPE_DIM = MAIN_DIM - ROPE_DIM      # 448
MIXED_ENTRY_BYTES = NOPE_DIM + 2 * ROPE_DIM   # 576


def mixed_quantize(x, nope_block: int = NOPE_DIM):
    """FP8 E4M3 nope dims with a float32 scale per block, BF16 rope dims.

    s = fl32(amax / 448) over each block of the first 448 dims; codes are
    E4M3(fl32(x / s)) (all zero when s == 0); the last 64 dims are stored as
    their BF16 bytes.  Returns (data [..., 576] uint8, scale [..., 448/blk]
    float32).
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == MAIN_DIM and NOPE_DIM % nope_block == 0
    nope = x[..., :NOPE_DIM].reshape(x.shape[:-1] + (NOPE_DIM // nope_block, nope_block))
    amax = np.abs(nope).max(axis=-1)
    s = np.float32(amax) / np.float32(E4M3_MAX)                 # float32
    with np.errstate(divide="ignore", invalid="ignore"):
        r = nope / s[..., None]
    codes = e4m3_encode(r)
    codes = np.where((s > 0)[..., None], codes, 0).astype(np.uint8)
    codes = codes.reshape(x.shape[:-1] + (NOPE_DIM,))
    rope = bf16_bytes(x[..., NOPE_DIM:])
    data = np.concatenate([codes, rope], axis=-1)
    return data, s.astype(np.float32)


def mixed_dequantize(data, scale, nope_block: int = NOPE_DIM) -> np.ndarray:
    data = np.asarray(data, dtype=np.uint8)
    scale = np.asarray(scale, dtype=np.float32).astype(np.float64)
    codes = data[..., :NOPE_DIM]
    v = e4m3_decode(codes).reshape(codes.shape[:-1] + (NOPE_DIM // nope_block, nope_block))
    v = (v * scale[..., None]).reshape(codes.shape)
    rope = bf16_from_bytes(data[..., NOPE_DIM:MIXED_ENTRY_BYTES])
    return np.concatenate([v, rope], axis=-1)


# ----------------------------------------------------- plane helpers ----

def quantize_entries(x, fmt: str, nope_block: int = NOPE_DIM):
    """Entry rows -> (data bytes, scale) of the plane format ``fmt``
    ('bf16', 'mixed', 'fp4', or 'fp4h': FP4 of the Hadamard-rotated 128-d
    indexer vector, see ``oracle/hadamard.py``)."""
    if fmt == "bf16":
        return bf16_bytes(x), None
    if fmt == "mixed":
        return mixed_quantize(x, nope_block)
    if fmt == "fp4":
        return fp4_quantize(x)
    if fmt == "fp4h":
        from .hadamard import fp4_quantize_hadamard
        return fp4_quantize_hadamard(x)
    raise ValueError(fmt)


def dequantize_entries(data, scale, fmt: str, nope_block: int = NOPE_DIM) -> np.ndarray:
    """float64 entry values of stored rows of the plane format ``fmt``."""
    if fmt == "bf16":
        return bf16_from_bytes(data)
    if fmt == "mixed":
        return mixed_dequantize(data, scale, nope_block)
    if fmt in ("fp4", "fp4h"):
        return fp4_dequantize(data, scale)   # fp4h: values in the rotated basis
    raise ValueError(fmt)

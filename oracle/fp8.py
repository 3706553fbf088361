"""8-bit (FP8 e4m3) storage of cached keys and values.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: Ultralytics glossary "PagedAttention", section "Related techniques"
(FP8 cache quantisation keeps keys and values at 8-bit precision, about
halving the cache against 16-bit formats).  The page names no format and no
scaling.
Readings taken, the plainest the rest supports:
* the 8-bit format is e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
  bits; exponent field 0 holds the subnormals m/8 * 2^-6; the all-ones
  pattern S.1111.111 is NaN and there is no infinity, so 448 is the largest
  finite value);
* each cached row (one token of one KV head, d values) carries its own fp32
  scale s = amax / 448 (s = 1 for an all-zero row), so that a token appended
  during decode never changes another token's codes;
* the code of a value x is the e4m3 value nearest to x / s, ties to the even
  code, saturating at +-448; x / s and amax / 448 are IEEE float32 divisions
  (the quantiser computes in fp32; the stored value is code * s).

Pinned in tests/test_oracle_pins.py against torch's float8_e4m3fn casts (all
256 codes decoded, random and midpoint values encoded), against the
round-trip error bound of the format, and against the saturation cases.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_NAN_CODES = (0x7F, 0xFF)


def e4m3_value(code: int) -> float:
    """The real number an e4m3 code stands for (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    if code in _NAN_CODES:
        return float("nan")
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# the 127 non-negative finite values in code order (codes 0x00 .. 0x7E)
_POS = np.array([e4m3_value(c) for c in range(0x7F)])


def e4m3_decode(codes) -> np.ndarray:
    """Codes (any integer array) -> float64 values."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    return np.array([e4m3_value(x) for x in c.ravel()]).reshape(c.shape)


def e4m3_decode_fast(codes) -> np.ndarray:
    """e4m3_decode by table lookup."""
    return E4M3_TABLE[np.asarray(codes).astype(np.int64) & 0xFF]


def e4m3_encode_one(x: float) -> int:
    """Nearest e4m3 code to x, ties to the even code, saturating at +-448."""
    x = float(x)
    if x != x:
        raise ValueError("NaN has no code here")
    sign = 0x80 if (x < 0 or (x == 0 and np.signbit(x))) else 0
    a = abs(x)
    if a >= E4M3_MAX:
        return sign | 0x7E
    # largest code whose value is <= a, then compare with the next one up
    lo = int(np.searchsorted(_POS, a, side="right")) - 1
    if _POS[lo] == a:
        return sign | lo
    hi = lo + 1
    dlo, dhi = a - _POS[lo], _POS[hi] - a
    if dlo < dhi or (dlo == dhi and lo % 2 == 0):
        return sign | lo
    return sign | hi


def e4m3_encode(x) -> np.ndarray:
    """e4m3_encode_one over an array, written with numpy: the same nearest
    value below and above, the same tie rule, the same saturation."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no code here")
    sign = np.where(np.signbit(x), 0x80, 0)
    a = np.abs(x)
    top = len(_POS) - 1                                  # code 0x7E = 448
    lo = np.clip(np.searchsorted(_POS, a, side="right") - 1, 0, top)
    hi = np.minimum(lo + 1, top)
    dlo, dhi = a - _POS[lo], _POS[hi] - a
    pick_lo = (dlo < dhi) | ((dlo == dhi) & (lo % 2 == 0)) | (lo == top)
    code = np.where(a >= E4M3_MAX, top, np.where(pick_lo, lo, hi))
    return (sign | code).astype(np.uint8)


# value of every code, for table lookups (NaN at the two NaN codes)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)])


def quantize_rows_fast(x):
    """quantize_rows with the per-row arithmetic vectorised over rows: the
    same float32 amax / 448 and x / scale, the same encoder."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1) if x.shape[-1] else np.zeros(x.shape[:-1], np.float32)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32),
                     np.float32(1.0)).astype(np.float32)
    q = (x / scale[..., None]).astype(np.float32)
    return e4m3_encode(q), scale


def quantize_row(x):
    """One cached row (float32-representable values, e.g. bf16) -> (codes
    uint8 [d], scale float32).  amax / 448 and x / scale in IEEE float32."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    q = (x32 / scale).astype(np.float32)
    return e4m3_encode(q), scale


def dequantize_row(codes, scale) -> np.ndarray:
    """float64 values the stored row stands for: code value times scale."""
    return e4m3_decode(codes) * float(scale)


def dequantize_rows(codes, scales) -> np.ndarray:
    """[..., d] codes and [...] scales -> float64 values."""
    return e4m3_decode_fast(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def quantize_rows(x):
    """[..., d] -> (codes [..., d] uint8, scales [...] float32), row by row."""
    x = np.asarray(x, dtype=np.float32)
    flat = x.reshape(-1, x.shape[-1])
    codes = np.empty(flat.shape, dtype=np.uint8)
    scales = np.empty(flat.shape[0], dtype=np.float32)
    for i in range(flat.shape[0]):
        codes[i], scales[i] = quantize_row(flat[i])
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1])

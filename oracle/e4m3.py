"""FP8 E4M3 codec restated from the OCP 8-bit floating point format definition.

TEST INFRASTRUCTURE: only tests, the smoke check and the benchmark's CPU
baseline use this module. The product path never imports it.

Format (OCP OFP8, E4M3 variant): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits. Exponent field 0 encodes subnormals m/8 * 2^-6. The pattern
S.1111.111 is NaN; there are no infinities, so the largest finite magnitude is
1.75 * 2^8 = 448.

The per-token quantisation recipe (one fp32 scale per cached c_KV row) is this
build's reading of the "MLA 之后，KV cache 确实得重新理解一遍" page, section
"所以 cache 逻辑到底哪里要重写", which says only that quantising c_kv spreads
the error over every head: scale = amax/448 in fp32 (1 when amax is 0, at
least FLT_MIN otherwise), code = round-to-nearest-even with saturation of
x/scale computed in fp32.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F
FLT_MIN = float(np.finfo(np.float32).tiny)


def decode_code(code: int) -> float:
    """Value of one E4M3 code from the bit fields."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# Table of all 256 codes, built from the bit-field definition above.
DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)
# Non-negative finite codes 0x00..0x7E in increasing value order.
_POS_VALUES = DECODE_TABLE[:0x7F]


def decode(codes: np.ndarray) -> np.ndarray:
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode_satfinite_rne(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code to each value, ties to the even code, saturating at 448.

    ``x`` is evaluated exactly in float64 (every fp32 value and every midpoint
    between E4M3 neighbours is exact there). NaN maps to the NaN code.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.int64)
    a_sat = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a_sat, side="left")      # first value >= a
    hi = np.clip(hi, 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = a_sat - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a_sat
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a_sat == _POS_VALUES[hi], hi, code)
    out = (code | sign).astype(np.uint8)
    out = np.where(np.isnan(x), NAN_CODE, out).astype(np.uint8)
    return out


def quantize_rows(x_f32: np.ndarray):
    """Per-row E4M3 quantisation in fp32 arithmetic: returns (codes uint8, scale fp32)."""
    x = np.asarray(x_f32, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    scale = np.where(scale < np.float32(FLT_MIN), np.float32(FLT_MIN), scale).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    return encode_satfinite_rne(y), scale


def dequantize_rows(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """e * scale rounded to fp32 (the stored cache value the attention sees), as float64."""
    v = decode(codes).astype(np.float32) * np.asarray(scale, np.float32)[..., None]
    return v.astype(np.float32).astype(np.float64)

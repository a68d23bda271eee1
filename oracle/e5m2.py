"""FP8 E5M2 codec, written out from the format's definition (float64 / integer NumPy).

vLLM stores the KV cache in FP8 as E4M3 or E5M2 ("量子化が vLLM の推論性能に与える影響",
section "KV キャッシュの量子化": vLLM は FP8 (E4M3 と E5M2) に対応).  The page prints no bit
layout; the reading taken is the IEEE-style FP8 E5M2 format: 1 sign bit, 5 exponent bits
with bias 15, 2 mantissa bits, S.11111.00 = infinity, S.11111.xx (xx != 0) = NaN,
largest finite magnitude 57344 (S.11110.11).  It is the upper byte of an IEEE binary16.

Encoding (reading R24) rounds to nearest with ties to the even mantissa over the whole
finite grid, subnormals included, saturates finite overflow and infinities to +-57344,
keeps the sign of zero, and encodes NaN as 0x7F.  Scaled quantisation follows the e4m3
rule of the cache write: e5m2(fl32(x * fl32(1/s))).
"""
from __future__ import annotations

import numpy as np

from .e4m3 import fl32, reciprocal_f32

E5M2_MAX = 57344.0
NAN_CODE = 0x7F


def decode(codes) -> np.ndarray:
    """Value of each e5m2 code (uint8 array) as float64; infinities and NaN included.

    Normal codes (exponent field e in 1..30): (-1)^s (1 + m/4) 2^(e-15).
    Subnormal codes (e == 0):                 (-1)^s (m/4) 2^-14.
    """
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 2) & 0x1F
    m = c & 0x3
    mag = np.where(e == 0, (m / 4.0) * 2.0 ** -14, (1.0 + m / 4.0) * np.exp2((e - 15).astype(np.float64)))
    mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    return np.where(s == 1, -mag, mag)


def decode_table() -> np.ndarray:
    """All 256 code values (index = code)."""
    return decode(np.arange(256, dtype=np.uint8))


def encode(y) -> np.ndarray:
    """Round float32 values to e5m2 codes (RNE, saturating at +-57344, NaN -> 0x7F).

    For a finite magnitude a < 57344 the grid spacing around a is 2^(e-2) with
    e = max(floor(log2 a), -14); a / 2^(e-2) is exact in float64 and numpy's ``round``
    breaks ties to even.  The code of n * 2^(e-2) is 4e + 56 + n (n == 8 lands on the
    next binade's first code; in the subnormal binade 4e + 56 = 0 and the code is n).
    """
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    neg = np.signbit(y)
    a = np.abs(y)
    nan = np.isnan(y)
    sat = (~nan) & (a >= E5M2_MAX)
    fin = (~nan) & (~sat)
    a_f = np.where(fin, a, 0.0)
    _, ex = np.frexp(a_f)
    e = np.where(a_f > 0, ex - 1, -14)
    e = np.maximum(e, -14)
    quantum = np.ldexp(1.0, (e - 2).astype(np.int64))
    n = np.round(a_f / quantum)
    code = (4 * e + 56 + n).astype(np.int64)
    code = np.where(n == 0, 0, code)
    code = np.where(sat, 0x7B, code)
    code = code | (neg.astype(np.int64) << 7)
    code = np.where(nan, NAN_CODE, code)
    return code.astype(np.uint8)


def quantize(x, scale) -> np.ndarray:
    """Scaled quantisation x -> e5m2(fl32(x * fl32(1/scale))), as for e4m3 (reading R3)."""
    inv = reciprocal_f32(scale)
    return encode(fl32(np.asarray(x, dtype=np.float64) * inv))


def dequantize(codes, scale) -> np.ndarray:
    """dec(code) * scale in float64."""
    return decode(codes) * np.asarray(scale, dtype=np.float64)

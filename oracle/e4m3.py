"""FP8 E4M3 codec, written out from the format's definition (float64 / integer NumPy).

The pages name e4m3 as the one format used throughout (vLLM blog "FP8 KV-Cache and
Attention quantization in vLLM", 引言: "本文全篇使用 e4m3 格式"); they do not print its
bit layout.  The reading taken here is the FP8 E4M3 ("fn") format: 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN,
largest finite magnitude 448 (S.1111.110).

Encoding rounds to nearest with ties to the even mantissa over the whole finite
grid, subnormals included, and saturates to +-448 (readings R1, R2: NaN -> 0x7F,
the sign of zero is kept).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def decode(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8 array) as float64; the two NaN codes give NaN.

    Normal codes (exponent field e > 0): (-1)^s (1 + m/8) 2^(e-7).
    Subnormal codes (e == 0):            (-1)^s (m/8) 2^-6.
    """
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    val = np.where(s == 1, -mag, mag)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def decode_table() -> np.ndarray:
    """All 256 code values (index = code)."""
    return decode(np.arange(256, dtype=np.uint8))


def encode(y) -> np.ndarray:
    """Round float32 values to e4m3 codes (RNE, saturating at +-448).

    ``y`` is taken as float32 (exactly representable in float64).  For a finite
    magnitude a < 448 the spacing of the e4m3 grid around a is 2^(e-3) with
    e = max(floor(log2 a), -6); a / 2^(e-3) is exact in float64 and numpy's
    ``round`` breaks ties to even, which is ties-to-even on the mantissa.
    The code of n * 2^(e-3) is 8e + 48 + n (n == 16 lands on the next binade's
    first code, n < 8 only occurs in the subnormal binade).
    """
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    neg = np.signbit(y)
    a = np.abs(y)
    nan = np.isnan(y)
    sat = (~nan) & (a >= E4M3_MAX)
    fin = (~nan) & (~sat)
    a_f = np.where(fin, a, 0.0)
    _, ex = np.frexp(a_f)
    e = np.where(a_f > 0, ex - 1, -6)
    e = np.maximum(e, -6)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))
    n = np.round(a_f / quantum)
    code = (8 * e + 48 + n).astype(np.int64)
    code = np.where(n == 0, 0, code)
    code = np.where(sat, 0x7E, code)
    code = code | (neg.astype(np.int64) << 7)
    code = np.where(nan, NAN_CODE, code)
    return code.astype(np.uint8)


def fl32(x) -> np.ndarray:
    """Round float64 values to the nearest float32 (returned as float64)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def reciprocal_f32(s) -> np.ndarray:
    """fl32(1/s) for float32 s.  1/s is first rounded to float64 and then to float32;
    that double rounding equals one correct rounding because 53 >= 2*24 + 2
    (Figueroa, "When is double rounding innocuous?", 1995)."""
    return fl32(1.0 / np.asarray(s, dtype=np.float32).astype(np.float64))


def quantize(x, scale) -> np.ndarray:
    """Scaled quantisation x -> e4m3(fl32(x * fl32(1/scale))) (reading R3: multiply by
    the round-to-nearest float32 reciprocal rather than divide).

    ``x`` holds bf16 (or float32) values as float64; the product of an 8- or 24-bit
    significand with a 24-bit one is exact in float64, so one rounding to float32
    follows.  ``scale`` broadcasts against ``x``.
    """
    inv = reciprocal_f32(scale)
    return encode(fl32(np.asarray(x, dtype=np.float64) * inv))


def dequantize(codes, scale) -> np.ndarray:
    """dec(code) * scale in float64."""
    return decode(codes) * np.asarray(scale, dtype=np.float64)

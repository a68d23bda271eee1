"""Pins of the oracle's e4m3 codec and scaled quantisation (CPU only).

The codec is checked against the format's definition by means that do not share its
arithmetic: hand-worked points (tests/golden/e4m3_points.txt), a brute-force nearest
search over the 254 finite codes for every bf16 bit pattern, round trips, and
torch's float8_e4m3fn cast as a library cross-check inside +-448.
"""
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _finite_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_decode_table_structure():
    t = e4m3.decode_table()
    fin = np.isfinite(t)
    assert fin.sum() == 254
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6 and t[0x38] == 1.0
    pos = t[0:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must be strictly increasing"
    for c in range(0x7F):
        assert t[c | 0x80] == -t[c] or (c == 0 and np.signbit(t[0x80]))
    # binade structure: 8 codes per exponent, spacing doubles every binade
    for e in range(1, 15):
        step = np.diff(t[8 * e: 8 * e + 8])
        assert np.allclose(step, 2.0 ** (e - 7 - 3))


def test_golden_points():
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            val, code = line.split()[:2]
            y = np.float32(float(val))
            got = int(e4m3.encode(np.array([y]))[0])
            assert got == int(code, 16), (val, hex(got), code)
            n += 1
    assert n >= 15


def _bruteforce_encode(y: float) -> int:
    """Nearest finite code by exhaustive search, ties to the code with even mantissa."""
    if np.isnan(y):
        return 0x7F
    if y >= 448.0:
        return 0x7E
    if y <= -448.0:
        return 0xFE
    best, best_d = None, None
    for c in _finite_codes():
        v = float(e4m3.decode(np.array([c], np.uint8))[0])
        d = abs(v - y)
        if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    # the two zeros: keep the input's sign
    if e4m3.decode(np.array([best], np.uint8))[0] == 0.0:
        return 0x80 if np.signbit(y) else 0x00
    return best


def test_encode_all_bf16_bruteforce():
    bits = np.arange(65536, dtype=np.uint32) << 16
    ys = bits.view(np.float32)
    got = e4m3.encode(ys)
    # vectorised brute force: distance to every finite code value
    codes = np.array(_finite_codes(), dtype=np.int64)
    vals = e4m3.decode(codes.astype(np.uint8))
    yy = ys.astype(np.float64)
    fin = np.isfinite(yy) & (np.abs(yy) < 448.0)
    d = np.abs(yy[fin, None] - vals[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    # among ties prefer the even code; among the two zeros prefer the input's sign
    score = cand * (1 + ((codes[None, :] & 1) == 0))
    choice = codes[np.argmax(score, axis=1)]
    zero = vals[np.argmax(score, axis=1)] == 0.0
    choice = np.where(zero, np.where(np.signbit(yy[fin]), 0x80, 0x00), choice)
    assert np.array_equal(got[fin].astype(np.int64), choice)
    # spot-check the scalar brute force on a sample (covers NaN / saturation too)
    rng = np.random.default_rng(0)
    for i in rng.choice(65536, 300, replace=False).tolist() + [0x7F80, 0xFF80, 0x7FC0, 0x43E0, 0xC3E8]:
        assert int(got[i]) == _bruteforce_encode(float(ys[i])), hex(i)
    # outside the finite range: saturation and NaN
    big = (~fin) & ~np.isnan(yy)
    assert np.all(got[big] == np.where(yy[big] > 0, 0x7E, 0xFE))
    assert np.all(got[np.isnan(yy)] == 0x7F)


def test_round_trip_every_code():
    for c in _finite_codes():
        v = e4m3.decode(np.array([c], np.uint8))
        assert int(e4m3.encode(v.astype(np.float32))[0]) == c
        # decode o encode o decode == decode
        assert e4m3.decode(e4m3.encode(v.astype(np.float32)))[0] == v[0]


def test_matches_torch_float8_inside_range():
    rng = np.random.default_rng(1)
    y = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 120.0)]).astype(np.float32)
    y = y[np.abs(y) < 448.0]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(y), ref)


def test_reciprocal_is_correctly_rounded_fp32():
    rng = np.random.default_rng(2)
    s = np.abs(rng.standard_normal(5000)).astype(np.float32) * np.float32(3.0) + np.float32(1e-3)
    ref = (np.float32(1.0) / s).astype(np.float64)     # IEEE single division
    assert np.array_equal(e4m3.reciprocal_f32(s), ref)


def test_quantize_unit_and_power_of_two_scales():
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal(4096).astype(np.float32) * 20).to(torch.bfloat16).float().numpy()
    x = x.astype(np.float64)
    assert np.array_equal(e4m3.quantize(x, np.float32(1.0)), e4m3.encode(x.astype(np.float32)))
    for k in (-3, 2, 5):
        s = np.float32(2.0 ** k)
        assert np.array_equal(e4m3.quantize(x, s), e4m3.encode((x * 2.0 ** -k).astype(np.float32)))


def test_quantize_reciprocal_not_division():
    # R3: x * fl32(1/s) is used, which differs from fl32(x / s) next to e4m3 rounding
    # ties.  Build inputs a few float32 ulps around every tie (times s) so that the
    # two readings part, and check that the oracle follows the reciprocal product.
    t = e4m3.decode_table()
    pos = np.sort(t[np.isfinite(t) & (t > 0)])
    ties = (pos[:-1] + pos[1:]) / 2
    s = np.float32(0.0123)
    xs = []
    for tie in ties:
        x0 = np.float32(tie * np.float64(s))
        for direction in (np.float32(np.inf), np.float32(-np.inf)):
            v = x0
            for _ in range(8):
                xs.append(v)
                v = np.nextafter(v, direction)
    xs = np.array(xs, dtype=np.float32)
    inv = np.float32(1.0) / s
    a = (xs * inv).astype(np.float32)
    div = (xs / s).astype(np.float32)
    assert np.any(e4m3.encode(a) != e4m3.encode(div)), "inputs must separate the two readings"
    assert np.array_equal(e4m3.quantize(xs.astype(np.float64), s), e4m3.encode(a))

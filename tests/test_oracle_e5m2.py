"""Pins of the oracle's e5m2 codec (CPU only): the decode against the IEEE binary16 whose
upper byte the code is, the encode against a brute-force nearest search over every bf16
pattern, round trips, saturation and NaN, and torch's float8_e5m2 cast inside the
finite range."""
import numpy as np
import torch

from oracle import e5m2


def test_decode_is_the_upper_byte_of_binary16():
    codes = np.arange(256, dtype=np.uint16)
    half = (codes << 8).astype(np.uint16).view(np.float16).astype(np.float64)
    got = e5m2.decode_table()
    assert np.array_equal(np.isnan(got), np.isnan(half))
    fin = ~np.isnan(half)
    assert np.array_equal(got[fin], half[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(half[fin]))
    assert got[0x7B] == 57344.0 and np.isinf(got[0x7C]) and got[0x01] == 2.0 ** -16


def _all_bf16_as_f32():
    bits = np.arange(65536, dtype=np.uint32) << 16
    return bits.astype(np.uint32).view(np.float32)


def test_encode_is_nearest_with_ties_to_even_over_every_bf16_value():
    y = _all_bf16_as_f32().astype(np.float64)
    got = e5m2.encode(y.astype(np.float32))
    tab = e5m2.decode_table()
    pos_codes = np.arange(0x7C)                 # +0 .. 57344
    pos_vals = tab[pos_codes]
    for i in np.flatnonzero(~np.isnan(y)):
        v = y[i]
        a = abs(v)
        if a >= 57344.0:
            want = 0x7B
        else:
            d = np.abs(pos_vals - a)
            cand = pos_codes[d == d.min()]
            want = int(cand[0]) if len(cand) == 1 else int([c for c in cand if c % 2 == 0][0])
        if np.signbit(v):
            want |= 0x80
        assert got[i] == want, (v, got[i], want)
    assert np.all(got[np.isnan(y)] == 0x7F)


def test_round_trip_and_saturation():
    codes = np.array([c for c in range(256) if (c & 0x7F) <= 0x7B], dtype=np.uint8)
    assert np.array_equal(e5m2.encode(e5m2.decode(codes).astype(np.float32)), codes)
    assert e5m2.encode(np.float32(np.inf)) == 0x7B and e5m2.encode(np.float32(-np.inf)) == 0xFB
    assert e5m2.encode(np.float32(1e30)) == 0x7B and e5m2.encode(np.float32(-0.0)) == 0x80


def test_matches_torch_float8_e5m2_inside_the_finite_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-6, 4, 20000),
                        np.array([57000.0, -57343.0, 2.0 ** -17, 3 * 2.0 ** -17])]).astype(np.float32)
    x = x[np.abs(x) < 57344.0]
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(e5m2.encode(x), ref)


def test_scaled_quantisation_with_power_of_two_scales_is_the_codec():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(1000) * 100.0
    for s in (1.0, 0.25, 8.0):
        assert np.array_equal(e5m2.quantize(x, np.float32(s)), e5m2.encode((x / s).astype(np.float32)))

"""Pins of the oracle's FP8 E4M3 codec and per-token quantiser (CPU only).

The codec is pinned to things outside the oracle: PyTorch's float8_e4m3fn
type (a library routine), the format's published landmark values (OCP 8-bit
floating point spec: bias 7, max 448, min normal 2^-6, min subnormal 2^-9,
S.1111.111 = NaN, no infinities) and exhaustive round-trip / tie properties.
"""
import math

import numpy as np
import pytest
import torch

import oracle

ALL = np.arange(256, dtype=np.uint8)
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_decode_all_codes_match_torch():
    dec = oracle.e4m3_decode_all()
    ref = torch_decode(ALL)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(dec), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(dec[~nan], ref[~nan])


def test_decode_landmarks():
    dec = oracle.e4m3_decode_all()
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6 and dec[0x07] == 7 * 2.0 ** -9
    assert dec[0x38] == 1.0 and dec[0xB8] == -1.0 and dec[0x00] == 0.0
    assert math.copysign(1.0, dec[0x80]) == -1.0 and dec[0x80] == 0.0
    # magnitudes strictly increase with the code over 0x00..0x7E
    assert np.all(np.diff(dec[:0x7F]) > 0)


def test_encode_round_trip_every_finite_code():
    dec = oracle.e4m3_decode_all()
    v = dec[FINITE].astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(v), FINITE)


def test_encode_midpoints_tie_to_even():
    dec = oracle.e4m3_decode_all()
    for c in range(0, 0x7E):
        lo, hi = dec[c], dec[c + 1]
        mid = np.float32((lo + hi) / 2)  # exact: at most 5 significant bits
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode([mid])[0] == even, hex(c)
        assert oracle.e4m3_encode([-mid])[0] == (even | 0x80)
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1e9))
        assert oracle.e4m3_encode([below])[0] == c
        assert oracle.e4m3_encode([above])[0] == c + 1


def test_encode_saturation_and_signed_zero():
    big = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    tiny = np.array([0.0, 2.0 ** -11, 2.0 ** -10], dtype=np.float32)  # 2^-10: tie -> even 0
    assert np.all(oracle.e4m3_encode(tiny) == 0x00)
    assert np.all(oracle.e4m3_encode(-tiny) == 0x80)
    assert oracle.e4m3_encode([np.nextafter(np.float32(2.0 ** -10), np.float32(1))])[0] == 0x01


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * 40,
        (rng.random(200_000).astype(np.float32) - 0.5) * 896,
        rng.standard_normal(50_000).astype(np.float32) * 2.0 ** -7,
    ])
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v)
    # torch keeps -0 as 0x80 too; compare every byte
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ quantiser
def test_quantiser_closed_form_grid():
    dec = oracle.e4m3_decode_all()
    rng = np.random.default_rng(3)
    for c in (1.25, 2.0 ** -7, 3.0):
        codes = rng.choice(FINITE, size=(64, 128)).astype(np.uint8)
        codes[:, 5] = 0x7E  # the row maximum is exactly 448 * c
        v = (dec[codes] * c).astype(np.float32)
        assert np.array_equal(v.astype(np.float64), dec[codes] * c)  # exact in fp32
        got, sc = oracle.quantize_rows(v)
        assert np.all(sc == np.float32(c))
        # -0 codes (0x80) decode to 0 and re-encode as +0 (v == +0.0 after the multiply by c>0
        # keeps the sign), so compare decoded values
        assert np.array_equal(dec[got], dec[codes])


def test_quantiser_zero_row_and_sign_symmetry():
    z = np.zeros((2, 64), dtype=np.float32)
    codes, sc = oracle.quantize_rows(z)
    assert np.all(codes == 0) and np.all(sc == 0)
    rng = np.random.default_rng(5)
    v = rng.standard_normal((100, 128)).astype(np.float32)
    c1, s1 = oracle.quantize_rows(v)
    c2, s2 = oracle.quantize_rows(-v)
    assert np.array_equal(s1, s2)
    assert np.array_equal(c1 ^ 0x80, c2)
    # the largest |v| maps to +-448 exactly
    i = np.argmax(np.abs(v), axis=1)
    top = c1[np.arange(100), i]
    assert np.all((top & 0x7F) == 0x7E)


def test_quantiser_power_of_two_invariance():
    rng = np.random.default_rng(9)
    v = rng.standard_normal((50, 64)).astype(np.float32)
    c1, s1 = oracle.quantize_rows(v)
    for k in (-8, 3, 20):
        c2, s2 = oracle.quantize_rows(v * np.float32(2.0 ** k))
        assert np.array_equal(c1, c2)
        assert np.array_equal(s2, s1 * np.float32(2.0 ** k))


def test_quantiser_matches_torch_restatement():
    rng = np.random.default_rng(11)
    v = rng.standard_normal((500, 128)).astype(np.float32) * rng.random((500, 1)).astype(np.float32) * 10
    codes, sc = oracle.quantize_rows(v)
    t = torch.from_numpy(v)
    amax = t.abs().amax(dim=1, keepdim=True)
    s = amax / 448.0
    ref = (t / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(sc, s[:, 0].numpy())
    assert np.array_equal(codes, ref)

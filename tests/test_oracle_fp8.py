"""Pins for the oracle's FP8 E4M3 codec and the Hadamard-rotated per-block
quantiser of the FP8 indexer ("GLM-5.2 / 总览" sub-doc index row 02:
"FP8 per-block + Hadamard"; glossary: KV FP8 is E4M3).  Code values come from
the OCP 8-bit floating point format, stored in tests/golden/e4m3_values.json.
"""
import json
import os

from fractions import Fraction as F

import numpy as np
import pytest
import scipy.linalg

import oracle
from synth import f32_to_bf16_bits, bf16_bits_to_f32

GOLD = os.path.join(os.path.dirname(__file__), "golden", "e4m3_values.json")


def test_spec_values_decode():
    g = json.load(open(GOLD))
    for code, val in g["values"]:
        got = oracle.e4m3_decode([int(code, 16)])[0]
        assert got == val and np.signbit(got) == np.signbit(val)
    for code in g["nan_codes"]:
        assert np.isnan(oracle.e4m3_decode([int(code, 16)])[0])


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes)
    assert np.array_equal(oracle.e4m3_encode(vals.astype(np.float32)), codes)
    pos = vals[codes < 0x80]
    assert (np.diff(pos) > 0).all()              # codes 0x00..0x7E increase


def test_round_to_nearest_even_and_saturation():
    codes = np.arange(0x00, 0x7E, dtype=np.uint8)
    lo = oracle.e4m3_decode(codes)
    hi = oracle.e4m3_decode(codes + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)   # midpoints exact in fp32
    got = oracle.e4m3_encode(mid)
    want = np.where(codes % 2 == 0, codes, codes + 1)
    assert np.array_equal(got, want)
    just_above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(oracle.e4m3_encode(just_above), codes + 1)
    assert oracle.e4m3_encode(np.float32([449, 1e6, 3e38, -500]))[:].tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert oracle.e4m3_encode(np.float32([np.nan]))[0] == 0x7F
    assert oracle.e4m3_encode(np.float32([2.0 ** -11, -2.0 ** -10]))[:].tolist() == [0x00, 0x80]


def test_hadamard_is_sylvester_and_orthonormal():
    H = scipy.linalg.hadamard(128).astype(np.float64) / np.sqrt(128)
    rng = np.random.default_rng(0)
    for _ in range(4):
        v = rng.standard_normal(128)
        hv = oracle.hadamard128_f64(v)
        assert np.allclose(hv, H @ v, rtol=0, atol=1e-12)
        assert np.allclose(oracle.hadamard128_f64(hv), v, rtol=0, atol=1e-12)  # H = H^T = H^-1
        u = rng.standard_normal(128)
        assert oracle.hadamard128_f64(u) @ hv == pytest.approx(u @ v, abs=1e-12)


def test_rotation_rows_exact_on_integers():
    # integer inputs: H x is an exact integer vector, divided once by sqrt(128)
    Hs = scipy.linalg.hadamard(128).astype(np.int64)
    rng = np.random.default_rng(1)
    xi = rng.integers(-100, 101, (5, 128))
    y = oracle.fp8_rotate_rows(f32_to_bf16_bits(xi.astype(np.float32)))
    want = (xi @ Hs.T).astype(np.float64) / np.sqrt(128.0)
    assert np.array_equal(y, want)
    e = np.zeros((1, 128), np.float32)
    e[0, 37] = 1
    assert np.array_equal(oracle.fp8_rotate_rows(f32_to_bf16_bits(e))[0], Hs[:, 37] / np.sqrt(128.0))


def _nearest_code(q):
    """Brute force over every finite E4M3 code: the one whose value is
    nearest to the exact rational q (ties: the even code)."""
    best = None
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        d = abs(q - F(float(oracle.e4m3_decode(np.array([c], np.uint8))[0])))
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def _nearest_f32(q):
    """The fp32 number nearest to the exact rational q > 0 (ties: even)."""
    r = np.float32(float(q))
    cands = [np.nextafter(r, np.float32(-np.inf)), r, np.nextafter(r, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(q - F(float(c))), int(np.float32(c).view(np.uint32)) & 1))


def test_quantiser_matches_exact_arithmetic():
    # scale = the fp32 nearest to amax/448 and every code = the E4M3 value
    # nearest to y/scale, both checked with exact rationals (y is the oracle's
    # fp64 rotation, pinned above against scipy's Hadamard)
    rng = np.random.default_rng(5)
    x = f32_to_bf16_bits(rng.standard_normal((3, 128)).astype(np.float32) / np.sqrt(128))
    x[2, 64:] = 0  # half a block
    q, s = oracle.fp8_quantize_rows(x)
    y = oracle.fp8_rotate_rows(x)
    for r in range(3):
        amax = F(float(np.abs(y[r]).max()))
        assert F(float(s[r])) == F(float(_nearest_f32(amax / 448)))
        for j in range(0, 128, 3):  # every third element keeps the brute force quick
            assert q[r, j] == _nearest_code(F(float(y[r, j])) / F(float(s[r]))), (r, j)


def test_quantiser_hand_worked_blocks():
    # one-hot block: H e_0 / sqrt(128) is the constant 1/sqrt(128): every
    # element is the block maximum, encoded as 448
    e0 = np.zeros((1, 128), np.float32)
    e0[0, 0] = 1.0
    q, s = oracle.fp8_quantize_rows(f32_to_bf16_bits(e0))
    assert s[0] == np.float32(1 / (448 * np.sqrt(128))) and (q[0] == 0x7E).all()
    # e_0 - e_1: rows i of H with (-1)^i -> 2/sqrt(128) at odd i, 0 at even i
    v = np.zeros((1, 128), np.float32)
    v[0, 0], v[0, 1] = 1.0, -1.0
    q, s = oracle.fp8_quantize_rows(f32_to_bf16_bits(v))
    assert s[0] == np.float32(2 / (448 * np.sqrt(128)))
    assert (q[0, 1::2] == 0x7E).all() and (q[0, 0::2] == 0x00).all()
    # a negated block gives sign-flipped codes and the same scale
    q2, s2 = oracle.fp8_quantize_rows(f32_to_bf16_bits(-v))
    assert s2[0] == s[0] and (q2[0, 1::2] == 0xFE).all()


def test_encode_decides_from_the_double():
    # the quantiser encodes fp64 quotients: a value just above a midpoint
    # (closer than fp32 resolves) rounds up, the midpoint itself to even
    assert oracle.e4m3_encode(np.array([1.0625]))[0] == 0x38
    assert oracle.e4m3_encode(np.array([1.0625 + 2.0 ** -40]))[0] == 0x39
    assert oracle.e4m3_encode(np.array([np.float32(1.0625 + 2.0 ** -40)]))[0] == 0x38


def test_quantiser_scale_codes_and_error_bound():
    rng = np.random.default_rng(2)
    x = f32_to_bf16_bits(rng.standard_normal((64, 128)).astype(np.float32) / np.sqrt(128))
    x[5] = 0                                     # an all-zero block
    q, s = oracle.fp8_quantize_rows(x)
    H = scipy.linalg.hadamard(128).astype(np.float64) / np.sqrt(128)
    xr = bf16_bits_to_f32(x).astype(np.float64) @ H.T
    assert s[5] == 1.0 and (q[5] == 0).all()
    for r in range(64):
        if r == 5:
            continue
        amax = np.abs(xr[r]).max()
        assert s[r] == pytest.approx(amax / 448, rel=1e-6)
        assert (q[r] & 0x7F).max() == 0x7E       # the block maximum lands on 448
        deq = oracle.e4m3_decode(q[r]) * np.float64(s[r])
        err = np.abs(deq - xr[r])
        # E4M3: 3 mantissa bits -> half-ulp 2^-4 relative on normals; subnormal
        # spacing 2^-9 * scale
        bound = np.maximum(np.abs(xr[r]) * 2.0 ** -4, 2.0 ** -10 * s[r]) * (1 + 1e-5) + 1e-7 * amax
        assert (err <= bound).all()


def test_rotation_preserves_indexer_dot_products():
    rng = np.random.default_rng(3)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    assert oracle.hadamard128_f64(q) @ oracle.hadamard128_f64(k) == pytest.approx(q @ k, abs=1e-12)

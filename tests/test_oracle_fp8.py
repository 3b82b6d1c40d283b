"""Pins for the oracle's FP8 E4M3 codec and the Hadamard-rotated per-block
quantiser of the FP8 indexer ("GLM-5.2 / 总览" sub-doc index row 02:
"FP8 per-block + Hadamard"; glossary: KV FP8 is E4M3).  Code values come from
the OCP 8-bit floating point format, stored in tests/golden/e4m3_values.json.
"""
import json
import os

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


def test_fast_transform_is_exact_on_integers():
    Hs = scipy.linalg.hadamard(128).astype(np.float64)
    rng = np.random.default_rng(1)
    v = rng.integers(-100, 101, 128).astype(np.float32)
    assert np.array_equal(oracle.fwht128_f32(v).astype(np.float64), Hs @ v.astype(np.float64))
    e = np.zeros(128, np.float32)
    e[37] = 1
    assert np.array_equal(oracle.fwht128_f32(e), Hs[:, 37].astype(np.float32))


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

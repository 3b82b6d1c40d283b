"""Pins of the oracle's interleaved RoPE and its fp64 -> bf16 rounding.

The rounding is pinned by exhaustive round trips, midpoints (ties to even)
and overflow; the rotation by position 0 (identity), a hand-worked vector,
the copied tail, the defining relative-position property of RoPE
(q(m).k(n) depends on m - n only), norm preservation and composition of
rotations (both within the bf16 rounding of the outputs)."""
import numpy as np

import oracle
import synth

THETA = 8e6  # GLM-5.2's rope_theta


def _bf16_value(bits):
    return synth.bf16_bits_to_f32(np.asarray([bits], np.uint16))[0]


def test_f64_to_bf16_round_trips_every_finite_bf16():
    for h in range(0, 1 << 16, 7):  # every 7th pattern, both signs, all exponents
        if (h & 0x7F80) == 0x7F80:
            continue  # inf / nan
        v = float(_bf16_value(h))
        got = oracle.f64_to_bf16(v)
        assert got == h or (v == 0.0 and (got & 0x7FFF) == 0), hex(h)


def test_f64_to_bf16_midpoints_and_neighbours():
    for h in (0x3F80, 0x3F81, 0x4049, 0x0080, 0x7F7E, 0xC2F3):
        a, b = float(_bf16_value(h)), float(_bf16_value(h + 1))
        mid = (a + b) / 2  # exact in fp64
        even = h if h % 2 == 0 else h + 1
        assert oracle.f64_to_bf16(mid) == even
        assert oracle.f64_to_bf16(np.nextafter(mid, a)) == h
        assert oracle.f64_to_bf16(np.nextafter(mid, b)) == h + 1
    assert oracle.f64_to_bf16(1e39) == 0x7F80 and oracle.f64_to_bf16(-1e39) == 0xFF80
    assert oracle.f64_to_bf16(float(_bf16_value(0x7F7F))) == 0x7F7F


def test_inv_freq():
    f = oracle.rope_inv_freq(THETA)
    assert f.shape == (32,) and f[0] == 1.0
    assert np.allclose(f[1:] / f[:-1], THETA ** (-2 / 64), rtol=1e-14)


def test_rope_identity_at_position_zero_and_copied_tail():
    rng = np.random.default_rng(1)
    x = synth.f32_to_bf16_bits(rng.standard_normal((5, 128)).astype(np.float32))
    f = oracle.rope_inv_freq(THETA)
    assert np.array_equal(oracle.rope_bf16(x, np.zeros(5, np.int32), f), x)
    y = oracle.rope_bf16(x, np.array([1, 17, 1000, 65536, 1048575], np.int32), f)
    assert np.array_equal(y[:, 64:], x[:, 64:])


def test_rope_hand_worked():
    x = np.zeros((1, 128), np.float32)
    x[0, 0], x[0, 3] = 1.0, 1.0  # pair 0 = (1, 0), pair 1 = (0, 1)
    xb = synth.f32_to_bf16_bits(x)
    f = oracle.rope_inv_freq(THETA)
    y = oracle.rope_bf16(xb, np.array([1], np.int32), f)[0]
    a1 = f[1]  # angle of pair 1 at position 1
    assert y[0] == oracle.f64_to_bf16(np.cos(1.0)) and y[1] == oracle.f64_to_bf16(np.sin(1.0))
    assert y[2] == oracle.f64_to_bf16(-np.sin(a1)) and y[3] == oracle.f64_to_bf16(np.cos(a1))
    assert (y[4:] == 0).all()


def _vals(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def test_rope_relative_position_norm_and_composition():
    rng = np.random.default_rng(2)
    n = 64
    q = synth.f32_to_bf16_bits(rng.standard_normal((n, 128)).astype(np.float32))
    k = synth.f32_to_bf16_bits(rng.standard_normal((n, 128)).astype(np.float32))
    f = oracle.rope_inv_freq(THETA)
    m = rng.integers(0, 1 << 20, n).astype(np.int32)
    d = rng.integers(-5000, 5000, n).astype(np.int32)
    s = rng.integers(0, 1 << 19, n).astype(np.int32)
    nn = np.clip(m + d, 0, None).astype(np.int32)
    dot = lambda a, b: np.einsum("ij,ij->i", _vals(a)[:, :64], _vals(b)[:, :64])
    # q(m).k(n) = q(m+s).k(n+s): only the offset matters (bf16 outputs: loose bound)
    lhs = dot(oracle.rope_bf16(q, m, f), oracle.rope_bf16(k, nn, f))
    rhs = dot(oracle.rope_bf16(q, m + s, f), oracle.rope_bf16(k, nn + s, f))
    scale = np.linalg.norm(_vals(q)[:, :64], axis=1) * np.linalg.norm(_vals(k)[:, :64], axis=1)
    assert (np.abs(lhs - rhs) <= 2e-2 * scale).all()
    # rotations preserve each pair's norm (within bf16 rounding)
    y = _vals(oracle.rope_bf16(q, m, f))[:, :64].reshape(n, 32, 2)
    x = _vals(q)[:, :64].reshape(n, 32, 2)
    assert np.allclose(np.linalg.norm(y, axis=2), np.linalg.norm(x, axis=2), rtol=1e-2, atol=1e-6)
    # rotating by a then by b equals rotating by a + b (within two bf16 roundings)
    a = rng.integers(0, 1 << 18, n).astype(np.int32)
    b = rng.integers(0, 1 << 18, n).astype(np.int32)
    two = _vals(oracle.rope_bf16(oracle.rope_bf16(q, a, f), b, f))
    one = _vals(oracle.rope_bf16(q, a + b, f))
    assert np.abs(two - one).max() <= 2e-2 * np.abs(_vals(q)).max()

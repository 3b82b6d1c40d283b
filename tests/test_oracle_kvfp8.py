"""Pins of the oracle's FP8 KV row (656 B: 512 E4M3 codes in four 128-dim
groups, four fp32 scales amax/448, the bf16 RoPE key) and its dequantisation:
the byte layout, exact round trips on the E4M3 grid, a hand-worked group,
the all-zero group, the relative error bound of E4M3 rounding, and the
largest element of each group landing on +-448 * scale."""
import numpy as np

import oracle
import synth


def _scales(rows):
    return np.ascontiguousarray(rows[:, 512:528]).view(np.float32)


def test_layout_and_rope_bytes():
    rng = np.random.default_rng(1)
    kv = synth.f32_to_bf16_bits(rng.standard_normal((7, 576)).astype(np.float32))
    q = oracle.kv_fp8_quantize(kv)
    assert q.shape == (7, 656)
    assert np.array_equal(np.ascontiguousarray(q[:, 528:]).view(np.uint16), kv[:, 512:])
    vals = synth.bf16_bits_to_f32(kv)[:, :512].reshape(7, 4, 128)
    amax = np.abs(vals).max(axis=2)
    assert np.array_equal(_scales(q), (amax / np.float32(448)).astype(np.float32))
    d = oracle.kv_fp8_dequantize(q)
    assert np.array_equal(d[:, 512:], kv[:, 512:])


def test_hand_worked_group_and_zero_group():
    x = np.zeros((1, 576), np.float32)
    x[0, :4] = [448.0, -224.0, 1.0, 0.5]  # scale 1: every value is an E4M3 value
    x[0, 128:132] = [3.0, -1.5, 0.0, 0.0]  # scale 3/448
    # group 2 all zero -> scale 1; group 3: a single value
    x[0, 384] = -2.0
    kv = synth.f32_to_bf16_bits(x)
    q = oracle.kv_fp8_quantize(kv)
    sc = _scales(q)[0]
    assert sc[0] == 1.0 and sc[2] == 1.0
    assert sc[1] == np.float32(3.0) / np.float32(448.0)
    assert sc[3] == np.float32(2.0) / np.float32(448.0)
    assert q[0, 0] == 0x7E and q[0, 1] == 0xF6 and q[0, 2] == 0x38 and q[0, 3] == 0x30
    assert (q[0, 256:384] == 0).all()
    d = synth.bf16_bits_to_f32(oracle.kv_fp8_dequantize(q))[0]
    assert np.array_equal(d[:4], [448.0, -224.0, 1.0, 0.5])
    assert d[384] == -2.0 and d[129] == -1.5 and d[128] == 3.0
    assert (d[256:384] == 0).all()


def test_round_trip_exact_on_the_e4m3_grid():
    # every value = (E4M3 value) * 2^e with the group's largest at 448 * 2^e:
    # the scale is 2^e exactly and every code, hence every value, is exact
    codes = np.arange(256, dtype=np.uint8)
    grid = np.array([oracle.e4m3_decode(np.array([c], np.uint8))[0] for c in codes])
    grid = grid[np.isfinite(grid)]
    rng = np.random.default_rng(2)
    x = np.zeros((3, 576), np.float64)
    for r, e in enumerate((-6, 0, 5)):
        for g in range(4):
            v = rng.choice(grid, 128)
            v[0] = 448.0
            x[r, 128 * g: 128 * g + 128] = v * 2.0 ** e
    kv = synth.f32_to_bf16_bits(x.astype(np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(kv).astype(np.float64), x.astype(np.float32))
    d = oracle.kv_fp8_dequantize(oracle.kv_fp8_quantize(kv))
    assert np.array_equal(d[:, :512], kv[:, :512])


def test_error_bound_and_group_maximum():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 576)).astype(np.float32) * np.float32(0.3)
    kv = synth.f32_to_bf16_bits(x)
    v = synth.bf16_bits_to_f32(kv)[:, :512].astype(np.float64).reshape(50, 4, 128)
    q = oracle.kv_fp8_quantize(kv)
    d = synth.bf16_bits_to_f32(oracle.kv_fp8_dequantize(q))[:, :512].astype(np.float64).reshape(50, 4, 128)
    sc = _scales(q).astype(np.float64)[:, :, None]
    # E4M3 keeps 3 mantissa bits: |x - q| <= 2^-4 |x| above its smallest normal
    # (2^-6 * scale), <= 2^-10 * scale below; then one bf16 rounding (2^-9)
    bound = np.maximum(np.abs(v) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 2 ** -8) + np.abs(v) * 2.0 ** -8
    assert (np.abs(d - v) <= bound).all()
    # the largest magnitude of each group is encoded as +-448
    i = np.abs(v).argmax(axis=2)
    codes = q[:, :512].reshape(50, 4, 128)
    top = np.take_along_axis(codes, i[:, :, None], axis=2)[:, :, 0]
    assert ((top & 0x7F) == 0x7E).all()


def _row(codes, scales):
    """An FP8 KV row built by hand: codes at dims 0.., the four group scales,
    a zero RoPE key."""
    r = np.zeros((1, 656), np.uint8)
    r[0, :len(codes)] = codes
    r[0, 512:528] = np.asarray(scales, np.float32).view(np.uint8)
    return r


def test_dequantisation_rounds_the_fp32_product():
    # code 0x3D = 1.625, scale 1 + 20165 * 2^-23 (exact in fp32): the exact
    # product is 1.625 + (2^15 + 1/8) * 2^-23, just above the midpoint
    # 1.625 + 2^-8 of the bf16 values 0x3FD0 / 0x3FD1.  The fp32 product
    # rounds down onto that midpoint, which rounds to the even 0x3FD0 (a
    # single rounding of the exact product would give 0x3FD1).
    s = np.float32(1 + 20165 * 2.0 ** -23)
    assert float(s) == 1 + 20165 * 2.0 ** -23
    assert np.float32(1.625) * s == np.float32(1.625 + 2.0 ** -8)
    d = oracle.kv_fp8_dequantize(_row([0x3D, 0xBD, 0x38], [s, 1, 1, 1]))[0]
    assert d[0] == 0x3FD0 and d[1] == 0xBFD0
    # 1.0 * s: fp32-exact, then s rounds to bf16 1.0 (0x3F80); zero codes stay zero
    assert d[2] == 0x3F80 and (d[3:512] == 0).all()
    # a product with no rounding at either step keeps every bit
    d2 = oracle.kv_fp8_dequantize(_row([0x7E, 0x01], [2.0 ** -3, 1, 1, 1]))[0]
    assert d2[0] == 0x4260 and d2[1] == 0x3980  # 448/8 = 56, 2^-9 / 8 = 2^-12


def test_codes_are_the_exact_quotients():
    # bf16 elements and group maxima for which the fp32 quotient x / scale
    # lands exactly on an E4M3 midpoint while the exact quotient lies just
    # above it: the definition (nearest E4M3 to x / scale) rounds up, where
    # an fp32 quotient followed by ties-to-even would round down.
    #   amax 1.375, x 0.2578125: x / scale = 84.0000018 -> 88 (fp32: 84 -> 80)
    #   amax 1.046875, x 0.003067: 1.31250004 -> 1.375  (fp32: 1.3125 -> 1.25)
    #   amax 1.40625, x 0.00824: 2.62500008 -> 2.75     (fp32: 2.625 -> 2.5)
    row = np.zeros((1, 576), np.uint16)
    row[0, [0, 1]] = [0x3FB0, 0x3E84]
    row[0, [128, 129]] = [0x3F86, 0x3B49]
    row[0, [256, 257]] = [0x3FB4, 0x3C07]
    q = oracle.kv_fp8_quantize(row)
    assert [int(q[0, 1]), int(q[0, 129]), int(q[0, 257])] == [0x6B, 0x3B, 0x43]
    assert oracle.e4m3_decode(q[0, [1, 129, 257]]).tolist() == [88.0, 1.375, 2.75]
    # the scales are the fp32 quotients amax / 448 (exact amax, one rounding)
    sc = _scales(q)[0]
    assert sc[0] == np.float32(1.375) / np.float32(448) and sc[3] == 1.0


def test_codes_nearest_by_brute_force():
    from fractions import Fraction as F
    rng = np.random.default_rng(9)
    kv = synth.f32_to_bf16_bits(rng.standard_normal((2, 576)).astype(np.float32) * np.float32(0.05))
    q = oracle.kv_fp8_quantize(kv)
    sc = _scales(q)
    x = synth.bf16_bits_to_f32(kv).astype(np.float64)
    grid = [(c, F(float(oracle.e4m3_decode(np.array([c], np.uint8))[0])))
            for c in range(256) if c not in (0x7F, 0xFF)]
    for r in range(2):
        for d in range(0, 512, 7):
            t = F(float(x[r, d])) / F(float(sc[r, d // 128]))
            best = min(grid, key=lambda cv: (abs(t - cv[1]), cv[0] & 1))[0]
            assert q[r, d] == best, (r, d)

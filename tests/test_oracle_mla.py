"""Pins for the oracle's absorbed sparse MLA.

Per head h and selected position s: z_s = scale * (q_lat . C[s,:512] +
q_rope . C[s,512:]); output sum_s softmax(z)_s C[s,:512]; the latent doubles
as key and value and the RoPE key enters only the score ("GLM-5.2 / 总览"
config table: KV = latent 512 + RoPE key 64; QK head dim 256 -> scale 1/16).
"""
import math

import numpy as np
import pytest

import oracle
from synth import f32_to_bf16_bits, bf16_bits_to_f32

DL, DR = 512, 64


def bf(x):
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def run(q_lat, q_rope, kv, idx, scale=1 / 16, key0=0):
    n = q_lat.shape[0]
    return oracle.sparse_mla(q_lat, q_rope, kv, np.arange(n, dtype=np.int32),
                             np.full(n, key0, np.int64), np.asarray(idx, np.int32), scale)


def rand_case(rng, n, H, rows, ints=True):
    if ints:
        g = lambda *s: bf(rng.integers(-3, 4, s))
    else:
        g = lambda *s: bf(rng.standard_normal(s) / 8)
    return g(n, H, DL), g(n, H, DR), g(rows, DL + DR)


def test_sparse_equals_dense_when_every_position_is_selected():
    rng = np.random.default_rng(0)
    H, rows = 4, 50
    ql, qr, kv = rand_case(rng, 3, H, rows, ints=False)
    pos = np.array([49, 20, 0], np.int32)
    K = 64
    idx = np.full((3, K), -1, np.int32)
    for i, p in enumerate(pos):
        idx[i, :p + 1] = rng.permutation(p + 1)    # all visible positions, any order
    o, l = run(ql, qr, kv, idx)
    od, ld = oracle.dense_mla(ql, qr, kv, np.arange(3, dtype=np.int32), pos,
                              np.zeros(3, np.int64), 1 / 16)
    assert np.allclose(o, od, rtol=0, atol=1e-12)
    assert np.allclose(l, ld, rtol=0, atol=1e-12)


def test_single_selected_position_returns_its_latent():
    rng = np.random.default_rng(1)
    ql, qr, kv = rand_case(rng, 1, 2, 10)
    idx = np.array([[-1, 7, -1, -1]], np.int32)
    o, l = run(ql, qr, kv, idx)
    c = bf16_bits_to_f32(kv[7]).astype(np.float64)
    assert np.array_equal(o[0, 0], c[:DL]) and np.array_equal(o[0, 1], c[:DL])
    z = (bf16_bits_to_f32(ql[0, 0]).astype(np.float64) @ c[:DL]
         + bf16_bits_to_f32(qr[0, 0]).astype(np.float64) @ c[DL:]) / 16
    assert l[0, 0] == pytest.approx(z, abs=1e-12)


def test_two_positions_closed_form_through_rope_only():
    # q_lat = 0: only the RoPE part scores; z_a - z_b = d -> weights sigmoid(d)
    kv = np.zeros((2, DL + DR), np.float32)
    kv[0, :DL] = 1.0
    kv[1, :DL] = -1.0
    kv[0, DL] = 2.0
    kv[1, DL] = 1.0
    q_lat = np.zeros((1, 1, DL), np.float32)
    q_rope = np.zeros((1, 1, DR), np.float32)
    q_rope[0, 0, 0] = 4.0                       # z = 4*C[s,512]/16 -> 0.5, 0.25
    o, l = run(bf(q_lat), bf(q_rope), bf(kv), [[0, 1]])
    pa = 1 / (1 + math.exp(-(0.5 - 0.25)))
    assert np.allclose(o[0, 0], pa * 1 + (1 - pa) * -1, rtol=0, atol=1e-12)
    assert l[0, 0] == pytest.approx(math.log(math.exp(0.5) + math.exp(0.25)), abs=1e-12)
    # equal scores: plain mean, lse = z + ln 2
    kv[1, DL] = 2.0
    o, l = run(bf(q_lat), bf(q_rope), bf(kv), [[0, 1]])
    assert np.allclose(o[0, 0], 0.0, atol=1e-12)
    assert l[0, 0] == pytest.approx(0.5 + math.log(2), abs=1e-12)


def test_weights_sum_to_one_and_scale_zero_is_a_mean():
    rng = np.random.default_rng(2)
    ql, qr, kv = rand_case(rng, 2, 3, 30)
    kvc = kv.copy()
    kvc[:, :DL] = bf(np.full(DL, 1.5))           # same latent everywhere
    idx = np.array([rng.choice(30, 9, replace=False), rng.choice(30, 9, replace=False)], np.int32)
    o, _ = run(ql, qr, kvc, idx)
    assert np.allclose(o, 1.5, rtol=0, atol=1e-12)
    o0, l0 = run(ql, qr, kv, idx, scale=0.0)
    for i in range(2):
        mean = bf16_bits_to_f32(kv[idx[i], :DL]).astype(np.float64).mean(0)
        assert np.allclose(o0[i], mean[None], rtol=0, atol=1e-12)
        assert np.allclose(l0[i], math.log(9), atol=1e-12)


def test_slot_order_and_padding_do_not_matter():
    rng = np.random.default_rng(3)
    ql, qr, kv = rand_case(rng, 1, 4, 40, ints=False)
    sel = rng.choice(40, 12, replace=False).astype(np.int32)
    a = run(ql, qr, kv, sel[None])
    b = run(ql, qr, kv, rng.permutation(sel)[None])
    padded = np.concatenate([sel, -np.ones(20, np.int32)])
    c = run(ql, qr, kv, rng.permutation(padded)[None])
    for x, y in ((a, b), (a, c)):
        assert np.allclose(x[0], y[0], rtol=0, atol=1e-12)
        assert np.allclose(x[1], y[1], rtol=0, atol=1e-12)


def test_empty_selection_gives_zero_and_neg_inf():
    rng = np.random.default_rng(4)
    ql, qr, kv = rand_case(rng, 1, 2, 5)
    o, l = run(ql, qr, kv, [[-1, -1]])
    assert (o == 0).all() and np.isneginf(l).all()


def test_latent_doubles_as_key_and_value():
    # changing only the RoPE key of a selected row changes the weights but the
    # output stays a convex combination of the latents
    rng = np.random.default_rng(5)
    ql, qr, kv = rand_case(rng, 1, 1, 6, ints=False)
    o, _ = run(ql, qr, kv, [[0, 1, 2, 3, 4, 5]])
    lat = bf16_bits_to_f32(kv[:, :DL]).astype(np.float64)
    assert (o[0, 0] <= lat.max(0) + 1e-12).all() and (o[0, 0] >= lat.min(0) - 1e-12).all()

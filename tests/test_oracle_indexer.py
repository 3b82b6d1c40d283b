"""Pins for the oracle's lightning-indexer scores.

I[t, s] = sum_j w[t, j] * ReLU(q[t, j] . k[s]) over 0 <= s <= pos[t], -inf
beyond ("GLM-5.2 / 总览" sub-doc index row 02: indexer with ReLU; config
table: 32 heads x 128 dims; "GLM-5.2架构与基准": causal selection among
earlier tokens).  Each test pins the oracle to a value worked out by hand or
fixed by a special case, never to a retyped copy of the formula.
"""
import numpy as np
import pytest

import oracle
from synth import f32_to_bf16_bits


def bf(x):
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def scores_of(q, w, k, pos, key0=0, max_len=None, **kw):
    q = np.asarray(q)
    nq = q.shape[0]
    rows = np.arange(nq, dtype=np.int32)
    pos = np.broadcast_to(np.asarray(pos, np.int32), (nq,))
    key0 = np.broadcast_to(np.asarray(key0, np.int64), (nq,))
    if max_len is None:
        max_len = int(pos.max()) + 1
    return oracle.indexer_scores(q, w, k, rows, pos, key0, max_len, **kw)


def test_hand_worked_two_heads():
    # heads j=0,1 of width 3; w = (0.5, -1)
    q = bf([[[1, -2, 0], [3, 1, 1]]])
    w = np.array([[0.5, -1.0]], np.float32)
    k = bf([[2, 1, 1],      # q0.k = 0 -> 0 ; q1.k = 8  -> -8          => -8
            [-1, 0, 2],     # q0.k = -1 -> 0; q1.k = -1 -> 0           => 0
            [3, 0, 5],      # q0.k = 3 -> 1.5; q1.k = 14 -> -14        => -12.5
            [9, 9, 9]])     # beyond pos=2                             => -inf
    got = scores_of(q, w, k, pos=2, max_len=4)
    assert got[0, :3].tolist() == [-8.0, 0.0, -12.5]
    assert got[0, 3] == -np.inf


def test_all_ones_closed_form():
    # q = k = 1, w = 1: every head contributes Di -> I = Hi * Di = 32 * 128
    q = bf(np.ones((1, 32, 128)))
    k = bf(np.ones((5, 128)))
    w = np.ones((1, 32), np.float32)
    got = scores_of(q, w, k, pos=4)
    assert (got == 4096.0).all()
    assert (scores_of(q, 2 * w, k, pos=4) == 8192.0).all()
    # negative dots are cut by the ReLU
    assert (scores_of(q, w, bf(-np.ones((5, 128))), pos=4) == 0.0).all()


def test_one_hot_head_is_a_relu_of_one_dot():
    q = np.zeros((1, 32, 128), np.float32)
    q[0, 5, 0] = 3.0
    w = np.zeros((1, 32), np.float32)
    w[0, 5] = 1.0
    k = np.zeros((5, 128), np.float32)
    k[:, 0] = np.arange(5) - 2          # q5.k = 3 (s - 2)
    got = scores_of(bf(q), w, bf(k), pos=4)
    assert got[0].tolist() == [0.0, 0.0, 0.0, 3.0, 6.0]


def test_causality_and_cache_offset():
    rng = np.random.default_rng(1)
    q = bf(rng.integers(-3, 4, (3, 32, 128)))
    w = rng.choice([-1.0, 0.0, 1.0, 2.0], (3, 32)).astype(np.float32)
    k = bf(rng.integers(-3, 4, (40, 128)))
    pos = np.array([5, 17, 39], np.int32)
    a = scores_of(q, w, k, pos, max_len=40)
    for i, p in enumerate(pos):
        assert np.isneginf(a[i, p + 1:]).all() and np.isfinite(a[i, :p + 1]).all()
    # keys beyond a row's position do not change that row
    k2 = k.copy()
    k2[6:] = bf(rng.integers(-3, 4, (34, 128)))
    b = scores_of(q, w, k2, pos, max_len=40)
    assert np.array_equal(a[0], b[0])
    # the same keys placed at cache row 100 give the same scores
    kbig = np.zeros((140, 128), np.uint16)
    kbig[100:] = k
    c = scores_of(q, w, kbig, pos, key0=100, max_len=40)
    assert np.array_equal(a, c)


def test_weight_linearity_and_head_permutation():
    rng = np.random.default_rng(2)
    q = bf(rng.integers(-3, 4, (2, 32, 128)))
    w = rng.choice([-1.0, 0.0, 1.0, 2.0], (2, 32)).astype(np.float32)
    k = bf(rng.integers(-3, 4, (16, 128)))
    a = scores_of(q, w, k, pos=15)
    assert np.array_equal(scores_of(q, -2 * w, k, pos=15), -2 * a)
    perm = rng.permutation(32)
    assert np.array_equal(scores_of(q[:, perm], w[:, perm], k, pos=15), a)
    # a head with a non-positive dot against every key contributes nothing
    w0 = w.copy()
    q0 = q.copy()
    q0[:, 7] = bf(np.zeros(128))
    w0[:, 7] = 1000.0
    q1 = q.copy()
    q1[:, 7] = bf(np.zeros(128))
    assert np.array_equal(scores_of(q0, w0, k, pos=15), scores_of(q1, w, k, pos=15))


def test_fp8_path_matches_bf16_on_exact_values():
    # E4M3 codes of small integers with unit scales reproduce the bf16 path
    codes = {-3: 0xC4, -2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44}
    rng = np.random.default_rng(3)
    qi = rng.integers(-3, 4, (2, 32, 128))
    ki = rng.integers(-3, 4, (12, 128))
    w = rng.choice([-1.0, 0.0, 1.0, 2.0], (2, 32)).astype(np.float32)
    enc = np.vectorize(codes.get)
    q8, k8 = enc(qi).astype(np.uint8), enc(ki).astype(np.uint8)
    ref = scores_of(bf(qi), w, bf(ki), pos=[11, 7], max_len=12)
    ones_q, ones_k = np.ones((2, 32), np.float32), np.ones(12, np.float32)
    got = scores_of(q8, w, k8, pos=[11, 7], max_len=12, dtype=1, q_scale=ones_q, k_scale=ones_k)
    assert np.array_equal(got, ref)
    # positive per-block scales factor out of the ReLU
    got2 = scores_of(q8, w, k8, pos=[11, 7], max_len=12, dtype=1, q_scale=4 * ones_q,
                     k_scale=0.25 * ones_k)
    assert np.array_equal(got2, ref)
    ks = np.linspace(0.5, 2.0, 12).astype(np.float32)
    got3 = scores_of(q8, w, k8, pos=[11, 7], max_len=12, dtype=1, q_scale=ones_q, k_scale=ks)
    fin = np.isfinite(ref)
    assert np.allclose(got3[fin], (ref * ks[None, :].astype(np.float64))[fin], rtol=0, atol=0)


def test_integer_scores_fit_fp32_exactly():
    # integer-valued workload bound: |I| <= 32 * 2 * 128 * 9 < 2^24
    assert 32 * 2 * 128 * 9 < 2 ** 24
    rng = np.random.default_rng(4)
    q = bf(rng.integers(-3, 4, (4, 32, 128)))
    w = rng.choice([-1.0, 0.0, 1.0, 2.0], (4, 32)).astype(np.float32)
    k = bf(rng.integers(-3, 4, (64, 128)))
    a = scores_of(q, w, k, pos=63)
    assert np.array_equal(a, a.astype(np.float32).astype(np.float64))
    assert np.array_equal(a, np.round(a))

"""The comparison rule for FP8 indexer codes (tests/fp8_rule.py), pinned on
the CPU: a single-precision Hadamard quantiser written independently here
(numpy float32, either stage order, normalised before or after the
butterfly) satisfies it with rare exceptions, and quantisers with plausible
mistakes (a wrong normalisation, a sign flipped in one butterfly stage, a
truncating encode, a wrong scale divisor) all violate it."""
import numpy as np
import pytest

import oracle
import synth
from fp8_rule import check_fp8_rows

STAGES = [1, 2, 4, 8, 16, 32, 64]


def _fwht32(v, order, flip_stage=None):
    n = v.shape[0]
    for h in order:
        w = v.reshape(n, 128 // (2 * h), 2, h)
        a, b = w[:, :, 0, :], w[:, :, 1, :]
        d = (b - a) if h == flip_stage else (a - b)
        v = np.stack([a + b, d], axis=2).reshape(n, 128).astype(np.float32)
    return v


def _quantise32(x_bits, order=STAGES, norm_first=False, norm=None, flip_stage=None, trunc=False,
                divisor=448.0):
    """fp32 quantiser: butterfly (float32 adds), normalising multiply, fp32
    amax / divisor, fp32 quotient, E4M3 round to nearest even (or toward
    zero when trunc)."""
    x = synth.bf16_bits_to_f32(np.asarray(x_bits).reshape(-1, 128)).astype(np.float32)
    c = np.float32(1 / np.sqrt(128)) if norm is None else np.float32(norm)
    if norm_first:
        y = _fwht32(x * c, order, flip_stage)
    else:
        y = _fwht32(x, order, flip_stage) * c
    amax = np.abs(y).max(1)
    sc = np.where(amax > 0, amax / np.float32(divisor), np.float32(1)).astype(np.float32)
    q = (y / sc[:, None]).astype(np.float32)
    codes = oracle.e4m3_encode(q)
    if trunc:
        over = np.abs(oracle.e4m3_decode(codes)) > np.abs(q.astype(np.float64))
        codes = np.where(over & ((codes & 0x7F) > 0), codes - 1, codes).astype(np.uint8)
    return codes, sc


def _rows(n=1500, seed=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 128)).astype(np.float32) / np.float32(np.sqrt(128))
    x[::97] *= np.float32(1e-3)     # small blocks
    x[5] = 0                        # an all-zero block
    x[7, :] = 0
    x[7, 3] = 1.0                   # one-hot: every rotated value is the maximum
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("order,norm_first", [(STAGES, False), (STAGES[::-1], False),
                                              (STAGES, True)])
def test_correct_fp32_quantisers_satisfy_the_rule(order, norm_first):
    x = _rows()
    codes, sc = _quantise32(x, order=order, norm_first=norm_first)
    r = check_fp8_rows(codes, sc, x, what="fp32 quantiser")
    assert r["code_exceptions"] <= 1e-3 * r["codes"]


@pytest.mark.parametrize("mistake", [dict(norm=1 / 8), dict(norm=1.0), dict(flip_stage=16),
                                     dict(trunc=True), dict(divisor=447.0)])
def test_plausible_mistakes_violate_the_rule(mistake):
    x = _rows()
    codes, sc = _quantise32(x, **mistake)
    with pytest.raises(AssertionError):
        check_fp8_rows(codes, sc, x, what=str(mistake))


def test_the_oracle_satisfies_its_own_rule_exactly():
    x = _rows(300, seed=4)
    q, s = oracle.fp8_quantize_rows(x)
    r = check_fp8_rows(q, s, x)
    assert r["code_exceptions"] == 0 and r["scale_exceptions"] == 0

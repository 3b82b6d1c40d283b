"""Comparison rule for FP8 indexer codes made by a single-precision quantiser.

The oracle quantises from the definition ("GLM-5.2 / 总览" sub-doc index row
02, "FP8 per-block + Hadamard"): y = H_128 x / sqrt(128) in fp64, scale = the
fp32 number nearest to max|y| / 448, code = the E4M3 value nearest to
y / scale.  A GPU quantiser that rotates in fp32 with a 7-stage butterfly
carries a bounded error, and near an E4M3 rounding boundary that error may
move a code by one step.  The rule below states that bound and allows such a
step only where the exact value lies within it of a boundary.

Error bound of an fp32 quantiser (u = 2^-24, the unit roundoff):
  * butterfly: at each of the 7 stages the nodes feeding output j cover
    disjoint groups of inputs, so their magnitudes sum to at most
    sum_i |x_i|; the rounding errors add up to <= 7 u sum_i |x_i| (to first
    order), and the normalising multiply by the fp32 value of 1/sqrt(128)
    adds <= 2 u |y_j|.  Taken as e_j = 8 u A + 3 u |y_j|, A = sum|x|/sqrt(128);
  * scale: amax moves by at most E = max_j e_j, and the fp32 division adds a
    rounding: |s_gpu - s_ref| <= E / 448 + 2.1 u s_ref (equality for an
    all-zero block, whose scale is 1);
  * code j: the GPU encodes fl32(y^_j / s_gpu), within
    band_j = e_j / s_gpu + |y_j| |1/s_gpu - 1/s_ref| + 1.1 u |v_j| of
    v_j = y_j / s_ref.  Its code's value must lie between the codes of
    v_j - band_j and v_j + band_j (equal to the oracle's code away from a
    boundary, one of the two neighbours of a boundary within band_j).

Exceptions (codes that differ from the oracle's) are counted; they must stay
rare (by default at most 1e-3 of the codes compared).
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

U = 2.0 ** -24


def check_fp8_rows(got_codes, got_scale, x_bits, max_exception_rate=1e-3, what=""):
    """Apply the rule to a GPU quantiser's output for bf16 rows x_bits
    [n, 128] (uint16 bit patterns).  Raises AssertionError on a violation;
    returns a dict with the counts."""
    x = np.ascontiguousarray(x_bits, np.uint16).reshape(-1, 128)
    n = x.shape[0]
    gc = np.ascontiguousarray(got_codes, np.uint8).reshape(n, 128)
    gs = np.asarray(got_scale, np.float32).reshape(n).astype(np.float64)
    rc, rs = oracle.fp8_quantize_rows(x)
    rs = rs.astype(np.float64)
    y = oracle.fp8_rotate_rows(x)
    A = np.abs(synth.bf16_bits_to_f32(x).astype(np.float64)).sum(1) / np.sqrt(128.0)
    e = 8 * U * A[:, None] + 3 * U * np.abs(y)
    E = e.max(1)
    zero = np.abs(y).max(1) == 0
    scale_ok = np.where(zero, gs == rs, np.abs(gs - rs) <= E / 448 + 2.1 * U * rs)
    bad_s = np.nonzero(~scale_ok)[0]
    assert bad_s.size == 0, (f"{what}: {bad_s.size} scales outside the bound, e.g. row {bad_s[0]}: "
                             f"got {gs[bad_s[0]]!r}, oracle {rs[bad_s[0]]!r}")
    v = y / rs[:, None]
    band = (e / gs[:, None] + np.abs(y) * np.abs(1 / gs - 1 / rs)[:, None] + 1.1 * U * np.abs(v))
    lo = oracle.e4m3_decode(oracle.e4m3_encode(v - band))
    hi = oracle.e4m3_decode(oracle.e4m3_encode(v + band))
    gv = oracle.e4m3_decode(gc)
    ok = (gv >= lo) & (gv <= hi)
    bad = np.argwhere(~ok)
    if bad.size:
        r, j = bad[0]
        raise AssertionError(
            f"{what}: {len(bad)} codes outside the band, e.g. row {r} dim {j}: got 0x{gc[r, j]:02x} "
            f"({gv[r, j]}), oracle 0x{rc[r, j]:02x}, exact value {v[r, j]!r} +- {band[r, j]:.3g}")
    exceptions = int((gc != rc).sum())
    assert exceptions <= max(1, max_exception_rate * gc.size), (
        f"{what}: {exceptions} of {gc.size} codes differ from the oracle's (all within the band, "
        f"but more than {max_exception_rate:g} of them)")
    return {"codes": int(gc.size), "code_exceptions": exceptions,
            "scale_exceptions": int((gs != rs).sum()), "rows": n}

"""Pins for the oracle's top-K selection.

The K positions with the largest scores among s <= pos; ties go to the lower
position; fewer than K visible positions are all taken and the rest padded
with -1 ("GLM-5.2 架构深度拆解" CH 2.2: keep the top 2048 positions; the
tie-break is this build's reading).  The oracle sorts; the pin below
characterises selection by rank instead: s is selected iff fewer than K
positions beat it, where s' beats s when its score is larger, or equal with
s' < s.
"""
import numpy as np
import pytest

import oracle


def brute_force(row, K):
    n = len(row)
    sel = []
    for s in range(n):
        beats = sum(1 for t in range(n) if row[t] > row[s] or (row[t] == row[s] and t < s))
        if beats < K:
            sel.append(s)
    return sel


@pytest.mark.parametrize("seed", range(6))
def test_rank_characterisation_with_many_ties(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 40, size=25).astype(np.int32)
    scores = np.full((25, 40), np.nan)
    for i, n in enumerate(lens):
        scores[i, :n] = rng.integers(-2, 3, n)    # five values: heavy ties
    for K in (1, 3, 8, 39, 64):
        got = oracle.topk(scores, lens, K)
        for i, n in enumerate(lens):
            want = brute_force(scores[i, :n], K)
            assert got[i, :len(want)].tolist() == want
            assert (got[i, len(want):] == -1).all()


def test_special_rows():
    n = 10
    const = np.zeros((1, n))
    assert oracle.topk(const, [n], 4)[0].tolist() == [0, 1, 2, 3]
    desc = -np.arange(n, dtype=np.float64)[None]
    assert oracle.topk(desc, [n], 3)[0].tolist() == [0, 1, 2]
    asc = np.arange(n, dtype=np.float64)[None]
    assert oracle.topk(asc, [n], 3)[0].tolist() == [7, 8, 9]
    # only the first len entries are candidates
    asc_inf = asc.copy()
    asc_inf[0, 6:] = 1e300
    assert oracle.topk(asc_inf, [6], 2)[0].tolist() == [4, 5]
    # K at least the visible length: everything, then -1 padding
    assert oracle.topk(asc, [4], 6)[0].tolist() == [0, 1, 2, 3, -1, -1]
    # -inf scores still count as candidates when visible
    m = np.array([[-np.inf, 1.0, -np.inf, -np.inf]])
    assert oracle.topk(m, [4], 2)[0].tolist() == [0, 1]


def test_gaussian_rows_match_a_full_sort():
    rng = np.random.default_rng(7)
    scores = rng.standard_normal((8, 300))
    lens = np.array([300, 299, 200, 65, 64, 63, 1, 150], np.int32)
    got = oracle.topk(scores, lens, 64)
    for i, n in enumerate(lens):
        order = np.argsort(-scores[i, :n], kind="stable")[:64]
        want = np.sort(order)
        assert got[i, :len(want)].tolist() == want.tolist()

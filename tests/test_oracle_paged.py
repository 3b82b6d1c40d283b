"""Pins of the oracle's paged-cache row map (paged_row, logical_cache): a
worked table by hand, the identity table (which must reduce to the
contiguous layout), unmapped blocks, and a random block permutation undone."""
import numpy as np

import oracle


def test_paged_row_worked_example():
    # two positions per block; sequence 0 owns blocks 3 then 0, sequence 1
    # owns blocks 1 then 2
    bt = np.array([[3, 0], [1, 2]])
    got = [[oracle.paged_row(bt, 2, b, s) for s in range(4)] for b in range(2)]
    assert got == [[6, 7, 0, 1], [2, 3, 4, 5]]
    assert oracle.paged_row(bt, 2, 0, 4) == -1                   # beyond the table
    assert oracle.paged_row(np.array([[0, -1]]), 2, 0, 3) == -1  # unmapped block
    assert oracle.paged_row(np.array([[0, -1]]), 2, 0, 1) == 1


def test_identity_table_is_contiguous():
    R, nb, lens = 128, 3, [300, 17, 384]
    bt = np.arange(len(lens) * nb).reshape(len(lens), nb)
    paged = np.arange(len(lens) * nb * R * 2).reshape(-1, 2)
    got = oracle.logical_cache(paged, bt, R, lens)
    want = np.concatenate([paged[b * nb * R: b * nb * R + n] for b, n in enumerate(lens)])
    assert np.array_equal(got, want)


def test_permuted_blocks_are_undone():
    rng = np.random.default_rng(3)
    R, lens = 4, [10, 3, 8]
    nblk = [(n + R - 1) // R for n in lens]
    total = sum(nblk) + 2
    ids = rng.permutation(total)
    bt = np.full((len(lens), max(nblk)), -1)
    logical = np.arange(sum(lens) * 3).reshape(-1, 3)  # unique rows
    paged = np.full((total * R, 3), -7)
    k, r0 = 0, 0
    for b, n in enumerate(lens):  # scatter block by block, the forward direction
        for j in range(nblk[b]):
            bt[b, j] = ids[k]
            m = min(R, n - j * R)
            paged[ids[k] * R: ids[k] * R + m] = logical[r0 + j * R: r0 + j * R + m]
            k += 1
        r0 += n
    assert np.array_equal(oracle.logical_cache(paged, bt, R, lens), logical)

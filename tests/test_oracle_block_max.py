"""Pins of the oracle's block maxima (the candidate source's block scores)
against values worked out by hand and against properties any block partition
of a row must have.  CPU only."""
import numpy as np

import oracle

NINF = -np.inf


def test_block_max_worked_by_hand():
    # row 0: keys 0..7 = 1, 5, 2, -inf, 3, 9, nan, 0 with ks = 0, ke = 7 and
    # blocks of 3: [0,3) -> max(1,5,2) = 5; [3,6) -> max(-inf,3,9) = 9;
    # [6,9) clipped to [6,7) holds only the NaN, which never wins -> -inf.
    x = np.array([[1, 5, 2, NINF, 3, 9, np.nan, 0]], np.float32)
    got = oracle.block_max(x, None, np.array([7], np.int32), 3)
    np.testing.assert_array_equal(got, [[5, 9, NINF]])
    # the same row with ks = 1, ke = 8 and blocks of 2 counted from ks:
    # [1,3) -> 5; [3,5) -> 3; [5,7) -> 9; [7,9) clipped to [7,8) -> 0.
    # (numbered from key 0 instead, the blocks would be 5, 2, 9, 0.)
    got = oracle.block_max(x, np.array([1], np.int32), np.array([8], np.int32), 2)
    np.testing.assert_array_equal(got, [[5, 3, 9, 0]])


def test_block_max_empty_and_single_block_rows():
    x = np.arange(20, dtype=np.float32).reshape(2, 10)
    # row 0 empty (ke = 0); row 1 one block covering [2, 10)
    got = oracle.block_max(x, np.array([0, 2], np.int32), np.array([0, 10], np.int32), 16)
    np.testing.assert_array_equal(got, [[NINF], [19]])


def test_block_max_partition_properties():
    rng = np.random.default_rng(11)
    rows, width = 7, 1000
    x = rng.standard_normal((rows, width)).astype(np.float32)
    x[rng.random((rows, width)) < 0.2] = NINF
    ke = rng.integers(0, width + 1, rows).astype(np.int32)
    ks = np.minimum(rng.integers(0, 200, rows), ke).astype(np.int32)
    for bs in (32, 64, 100, 128, 999, 5000):
        got = oracle.block_max(x, ks, ke, bs)
        assert got.shape == (rows, -(-width // bs))
        for r in range(rows):
            live = x[r, ks[r]:ke[r]]
            nb = -(-(ke[r] - ks[r]) // bs)
            # blocks past the row end hold nothing
            assert np.all(got[r, nb:] == NINF)
            # the blocks partition [ks, ke): the largest block score is the
            # row's largest logit, and it sits in the block of its argmax
            if live.size and np.isfinite(live).any():
                t = int(np.argmax(live))
                assert got[r].max() == live[t]
                assert got[r, t // bs] == live[t]
            # every key is at most its block's score
            for j in range(nb):
                seg = live[j * bs:(j + 1) * bs]
                assert np.all(seg <= got[r, j])

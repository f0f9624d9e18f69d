"""Pins for the THD packing oracle: a worked example written out by hand,
the round trip, and the lengths the packed-row workload generator uses."""
import numpy as np

from oracle import thd


def test_worked_example():
    x = np.arange(2 * 3 * 2).reshape(2, 3, 2)      # rows [[0,1],[2,3],[4,5]], [[6,7],...]
    y = thd.pack_thd(x, [2, 1])
    assert y.tolist() == [[0, 1], [2, 3], [6, 7]]
    assert thd.row_offsets([2, 1], 3).tolist() == [0, 2, 3]
    back = thd.unpack_bshd(y, [2, 1], 3)
    assert back.tolist() == [[[0, 1], [2, 3], [0, 0]], [[6, 7], [0, 0], [0, 0]]]


def test_clamping_and_empty_rows():
    x = np.ones((3, 4, 4), dtype=np.int32)
    assert thd.row_offsets([-3, 9, 0], 4).tolist() == [0, 0, 4, 4]
    assert thd.pack_thd(x, [-3, 9, 0]).shape == (4, 4)
    assert thd.pack_thd(x, [0, 0, 0]).shape == (0, 4)


def test_round_trip_random():
    rng = np.random.default_rng(5)
    x = rng.integers(0, 1000, size=(5, 37, 3, 4)).astype(np.int32)
    lens = rng.integers(0, 38, size=5)
    y = thd.pack_thd(x, lens)
    assert y.shape[0] == int(lens.sum())
    back = thd.unpack_bshd(y, lens, 37)
    for b in range(5):
        assert np.array_equal(back[b, :lens[b]], x[b, :lens[b]])
        assert not back[b, lens[b]:].any()
    assert np.array_equal(thd.pack_thd(back, lens), y)


def test_rows_keep_their_identity():
    """Each token row carries its (row, position); the packed order is row by
    row, positions ascending, and nothing from the padding."""
    B, S = 4, 9
    x = np.zeros((B, S, 4), dtype=np.int32)
    for b in range(B):
        for s in range(S):
            x[b, s] = (b, s, b * 100 + s, 7)
    lens = [3, 0, 9, 1]
    y = thd.pack_thd(x, lens)
    expect = [(b, s) for b in range(B) for s in range(lens[b])]
    assert [tuple(r[:2]) for r in y.tolist()] == expect

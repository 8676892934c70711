"""The persistent schedule of the tensor-core gradient passes, as restated in sched_util (CPU).

The stored-exponential dW pass keeps one copy of the scaled rows of h per segment of a 128-token
tile (the pairs of the one-pass kernel's schedule that share the tile) and has room for eight;
the schedule's rule that every pair covers at least a sixth of a tile bounds the count at seven.
Every tile's segments must also visit each vocabulary block exactly once, in the rotated order."""

import pytest

import sched_util as S

PAIRS = 76   # a 152-SM GB300


@pytest.mark.parametrize("V", [65, 100, 257, 1000, 3001, 50304])
def test_segments_per_tile_fit_the_copies(V):
    worst = 0
    for N in list(range(1, 2048, 37)) + [4096, 6000, 16384, 65536]:
        worst = max(worst, S.max_segments(N, V, PAIRS))
    assert worst <= 7


@pytest.mark.parametrize("N,V", [(16384, 50304), (65536, 50304), (300, 1000), (2000, 50304), (257, 100),
                                 (520, 3001)])
def test_segments_partition_each_tile_in_rotated_order(N, V):
    nblk = -(-V // S.YB)
    for t in range(-(-N // S.XT)):
        segs = S.segment_blocks(N, V, PAIRS, t)
        flat = [b for seg in segs for b in seg]
        assert sorted(flat) == list(range(nblk))
        r = S.rotation(N, V, PAIRS, t)
        assert flat == [(j + r) % nblk for j in range(nblk)]


def test_head_workload_has_two_segments_per_tile():
    # the 124M head (16,384 tokens, V = 50,304): a pair covers ~1.7 tiles, so a tile is shared
    # by at most two pairs and the dW pass reads two copies of the scaled rows
    assert S.max_segments(16384, 50304, PAIRS) == 2

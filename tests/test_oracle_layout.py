"""Oracle pins: block LUT and shard ranges.

"面向 Blockwise FP8 量化的 ZeRO 优化器设计" §块粒度切分: pad to multiples of 128,
record real and padded extents, shard on 128x128 block edges; §参数布局变换:
block order of view(E,R/128,128,C/128,128).permute(0,1,3,2,4)."""
import numpy as np
import pytest

import oracle
from tests._golden import parse_shapes, rows


@pytest.mark.parametrize("row", rows("layout_counts.txt"), ids=lambda r: f"{r[0]}-r{r[4]}")
def test_golden_counts_and_ranges(row):
    name, shapes, nblk, dp, rank, b0, b1 = row
    shapes = parse_shapes(shapes)
    assert oracle.count_blocks(shapes) == int(nblk)
    assert oracle.shard_range(int(nblk), int(dp), int(rank)) == (int(b0), int(b1))


def _coverage(shapes):
    """Brute force: mark every real element each LUT entry covers."""
    lut = oracle.build_lut(shapes)
    counts = [np.zeros((e, r, c), dtype=np.int32) for e, r, c in shapes]
    for k, (p, e, rb, cb, rr, cr) in enumerate(lut):
        E, R, C = shapes[p]
        # real extents agree with the padded-tile bounds
        assert 1 <= rr <= 128 and 1 <= cr <= 128
        assert rr == min(128, R - 128 * rb) and cr == min(128, C - 128 * cb)
        counts[p][e, 128 * rb:128 * rb + rr, 128 * cb:128 * cb + cr] += 1
    return lut, counts


@pytest.mark.parametrize("shapes", [
    [(1, 300, 200)],
    [(3, 129, 257), (1, 1, 1), (2, 128, 128), (1, 17, 690)],
    [(1, 5, 1000), (4, 250, 3)],
])
def test_lut_covers_every_real_element_once(shapes):
    lut, counts = _coverage(shapes)
    for c in counts:
        assert (c == 1).all()
    # block order: params in order, then (e, rb, cb) lexicographic
    keys = [tuple(x) for x in lut[:, :4]]
    assert keys == sorted(keys)
    assert len(lut) == oracle.count_blocks(shapes)


def test_ranges_tile_the_block_list():
    for nblk in [0, 1, 6, 7, 86016, 42574]:
        for dp in [1, 2, 3, 8, 13]:
            prev = 0
            for r in range(dp):
                b0, b1 = oracle.shard_range(nblk, dp, r)
                assert b0 == prev and b0 <= b1
                # element offset of every shard is a whole number of 128x128 blocks
                assert (b0 * 16384) % 16384 == 0
                prev = b1
            assert prev == nblk

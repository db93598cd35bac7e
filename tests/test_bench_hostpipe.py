"""Host-side layout of bench.py's end-to-end leg: how a step's inputs are packed into one pinned
buffer and how large copies are cut into pieces (no GPU needed)."""
import random

import bench


def test_pack_layout_aligned_and_disjoint():
    rng = random.Random(5)
    for _ in range(200):
        sizes = [rng.choice([0, 1, 3, 255, 256, 257, rng.randint(1, 1 << 20)]) for _ in range(rng.randint(1, 9))]
        offs, total = bench.pack_layout(sizes)
        assert all(o % 256 == 0 for o in offs)
        ends = [o + n for o, n in zip(offs, sizes)]
        assert all(ends[i] <= offs[i + 1] for i in range(len(sizes) - 1))  # in order, no overlap
        assert total == max(1, ends[-1])
        assert all(offs[i + 1] - ends[i] < 256 for i in range(len(sizes) - 1))  # padding only to the boundary


def test_copy_pieces_cover_in_order():
    for n in [1, 255, (16 << 20) - 1, 16 << 20, (32 << 20) + 7, 134244932, 1 << 30]:
        p = bench.copy_pieces(n)
        assert p[0][0] == 0 and p[-1][1] == n
        assert all(lo < hi for lo, hi in p)
        assert all(p[i][1] == p[i + 1][0] for i in range(len(p) - 1))
        assert all(lo % 256 == 0 for lo, _ in p)
        assert 1 <= len(p) <= 4
        if len(p) > 1:
            assert min(hi - lo for lo, hi in p) >= (16 << 20) - 256
    assert len(bench.copy_pieces(134217728)) == 4 and len(bench.copy_pieces(3674368)) == 1
